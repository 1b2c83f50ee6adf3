/*
 * kda.h -- C ABI of the GB300 (sm_103a) chunked Kimi Delta Attention (KDA) training library.
 *
 * The library computes, per head with head dim d = 128 and for documents packed back to back in
 * one sequence (boundaries given by cu_seqlens), the gated delta rule
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp(g_t)) S_{t-1} + beta_t k_t v_t^T,   o_t = scale * S_t^T q_t
 *
 * with the state S [key, value] reset at every document start (to h0 when given, else zero), its
 * reverse-mode gradient, and the fragment-summary / transfer-walk step that carries the state over
 * fragment boundaries of a long document.  It is evaluated chunk-parallel with chunks of 64 tokens
 * restarted at every document start.
 *
 * Sources (page title, section):
 *  - "fix(cake_kda_det): gate-gradient accuracy of the GLM intra stage (diagonal TF32 rounding)"
 *    (flashinfer PR #8909), summary: the chunked KDA training package computes forward and
 *    backward; gate form g (precomputed FP32 log gate) or raw (gate computed from A_log /
 *    dt_bias); Q/K L2 norm off or fused; backward from the saved forward set or by checkpoint
 *    replay (saved = None); bf16 q/k/v/beta, fp32 gate, head dim 128.  Same page, first commit
 *    message: the gate gradient flows on into dA_log and dt_bias.
 *  - "perf(cake_kda): auto grad, ship the BF16x3 half-width transfer walk on the context-parallel
 *    route" (flashinfer PR #7176), PR description: fragment state is passed as FP32 affine
 *    summaries and the transfer walk composes S_out = M * S_in + B; summary by CodeRabbit: a head
 *    count below one is rejected with a clear validation error.
 *  - "feat(cake_gqa_train): packed-varlen HD256 GQA training attention for SM100 / SM103 / SM107"
 *    (flashinfer PR #7774), file list: caller-held workspace reused across dynamic shapes, lengths
 *    read on the device only, no device synchronisation, launches on the caller's current stream.
 *
 * Conventions shared by every entry point
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The library allocates nothing,
 *    keeps no pointer after a call returns, and never synchronises the device: every call only
 *    enqueues kernels on `stream` (NULL = the legacy default stream).
 *  - Layouts are dense row-major ("THD"): q, k, v, dO are bf16 [T, H, 128]; beta is bf16 [T, H];
 *    o, dq, dk, dv [T, H, 128] and dbeta [T, H] are fp32 when kda_problem.out_fp32 = 1, else bf16
 *    (the outputs are heavy-tailed: bf16 storage alone puts max|err|/rms(ref) of o near 4e-2 on
 *    the raw-gate workloads, so fp32 is the parity-grade choice);
 *    g / a and dg / da are fp32 [T, H, 128]; A_log is fp32 [H];
 *    dt_bias, ddt_bias are fp32 [H, 128]; h0, ht, dht, dh0 are fp32 [N, H, 128, 128] indexed
 *    [key][value]; cu_seqlens is int32 [N + 1] on the device with cu_seqlens[0] = 0,
 *    non-decreasing, cu_seqlens[N] = T.  Empty documents are allowed (their ht = h0).
 *  - Every pointer must be 16-byte aligned.  Outputs are fully overwritten, never accumulated.
 *  - Errors found on the host are returned as a status and nothing is launched.  Errors found on
 *    the device (malformed cu_seqlens; in g form a gate value above 0) set a status word inside the
 *    workspace and make the kernels skip their work; read it with kda_read_device_status.  The library never aborts and never
 *    traps on the device.
 *  - Results are bitwise reproducible run to run (no floating-point atomics; every reduction has
 *    a fixed order), and a document's outputs do not depend on the other documents of the pack
 *    (except dA_log and ddt_bias, which are sums over all documents).
 */
#ifndef KDA_GB300_H
#define KDA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without pulling in the CUDA headers (same underlying type). */
typedef struct CUstream_st* kda_stream_t;

typedef enum kda_status {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size, H < 1, T < 0, N < 1 */
    KDA_ERR_UNSUPPORTED = 2,  /* d != 128, no sm_103 device, unsupported option */
    KDA_ERR_WORKSPACE = 3,    /* workspace (or saved buffer) smaller than the size query says */
    KDA_ERR_CUDA = 4,         /* a CUDA runtime call failed (launch error) */
    KDA_ERR_TIMEOUT = 5,      /* a bounded device-side wait gave up (reported via device status) */
    KDA_ERR_DEVICE_CHECK = 6, /* device-side validation failed (malformed cu_seqlens, g > 0) */
    KDA_ERR_TOO_LARGE = 7     /* problem needs more scratch than kda_fwd_static_ws holds */
} kda_status;

typedef enum kda_gate_form {
    KDA_GATE_G = 0,   /* g_or_a holds the per-channel fp32 log gate g, which must be <= 0 (a
                         decaying gate): a g > 0 or NaN inside a document sets the device status
                         KDA_ERR_DEVICE_CHECK and the call's later kernels write nothing */
    KDA_GATE_RAW = 1  /* g_or_a holds a; g = -exp(A_log[h]) * softplus(a + dt_bias[h]) */
} kda_gate_form;

typedef enum kda_op {
    KDA_OP_FWD = 0,         /* kda_fwd */
    KDA_OP_BWD_SAVED = 1,   /* kda_bwd with the saved forward set */
    KDA_OP_BWD_REPLAY = 2,  /* kda_bwd with saved == NULL (forward recomputed) */
    KDA_OP_FRAGMENT = 3,    /* kda_fragment_summary (either mode) */
    KDA_OP_WALK = 4         /* kda_transfer_walk (needs no workspace) */
} kda_op;

typedef enum kda_frag_mode {
    KDA_FRAG_FWD = 0, /* M (transition product) and B (state from zero) per fragment and head */
    KDA_FRAG_BWD = 1  /* C: gradient at the fragment start for zero end gradient */
} kda_frag_mode;

/* Problem description.  cu_seqlens is the only pointer in it and is read on the device only. */
typedef struct kda_problem {
    int64_t T;                  /* total packed tokens, >= 0 */
    int32_t N;                  /* documents (or fragments), 1 .. 65535 */
    int32_t H;                  /* heads, 1 .. 65535; N * H * 4 above INT32_MAX is
                                   KDA_ERR_UNSUPPORTED (one-dimensional recurrence grids) */
    int32_t d;                  /* head dim; must be 128 */
    int32_t gate;               /* kda_gate_form */
    int32_t l2norm;             /* 0: q, k used as given; 1: fused q/sqrt(|q|^2+eps), same for k */
    int32_t out_fp32;           /* 1: o, dq, dk, dv, dbeta are fp32; 0: they are bf16 */
    int32_t group_chunks;       /* 0: each document's state recurrence runs over its chunks in one
                                   serial chain.  G > 0: documents are cut into groups of G chunks
                                   (64 G tokens; the last group of a document may be shorter); the
                                   groups' affine state summaries (M, B) -- and in the backward the
                                   gradient summaries C -- are computed in parallel, the transfer
                                   walk (BF16x3, full width) composes them into each group's start
                                   state (start gradient), and the groups are finished in parallel.
                                   The serial chain shrinks from a document's chunks to G chunks
                                   plus a walk step per group.  Results equal the G = 0 ones up to
                                   rounding (not bitwise); for a given G they are bitwise
                                   reproducible and each document stays independent of the others.
                                   kda_fragment_summary and kda_fwd_static_ws take G = 0 only. */
    float scale;                /* output scale (1 for the plain recurrence) */
    float l2_eps;               /* eps of the fused L2 norm (1e-6) */
    const int32_t* cu_seqlens;  /* device int32 [N+1] */
} kda_problem;

/* Size query.  For op = KDA_OP_FWD it returns the workspace of kda_fwd and, in saved_bytes, the
 * size of the saved forward set that kda_fwd writes (when its `saved` argument is non-NULL) and
 * kda_bwd reads.  Sizes depend on T, N and H only (never on the lengths in cu_seqlens), so one
 * allocation serves every pack with the same T, N, H.  Either output pointer may be NULL. */
kda_status kda_workspace_size(const kda_problem* p, int op, size_t* ws_bytes, size_t* saved_bytes);

/* Forward.  Writes o ([T,H,128], fp32 or bf16 per out_fp32), ht (fp32 [N,H,128,128], nullable) and, when `saved` is
 * non-NULL, the saved forward set (per-chunk states and chunk write vectors) for kda_bwd.
 * h0 (nullable = zero initial state).  A_log / dt_bias are read only in raw gate form.
 * Source: the chunked KDA training package page (PR #8909), summary (forward pass, gate forms,
 * fused L2 norm). */
kda_status kda_fwd(const kda_problem* p, const void* q, const void* k, const void* v,
                   const void* beta, const float* g_or_a, const float* A_log,
                   const float* dt_bias, const float* h0, void* o, float* ht, void* saved,
                   void* ws, size_t ws_bytes, kda_stream_t stream);

/* Allocation-free forward for callers that cannot allocate device memory themselves -- e.g. code
 * that runs where the framework owns every device allocation and offers no workspace (a plugin
 * or op inside a host runtime), or code that must not grow the memory footprint behind the
 * caller's allocator.  It computes exactly what kda_fwd computes with saved == NULL (o and,
 * when non-NULL, ht), but its scratch lives in one static device array inside this library:
 * KDA_STATIC_WS_BYTES (64 MiB) on every GPU that loads the library, held until the process exits.
 * The pages describe no such entry point; it has no counterpart there.
 *  - Problems whose kda_fwd workspace (kda_workspace_size, KDA_OP_FWD) exceeds
 *    KDA_STATIC_WS_BYTES are rejected with KDA_ERR_TOO_LARGE before anything is launched
 *    (roughly: (ceil(T/64) + N) * H <= 300 (chunk, head) pairs, e.g. 4096 tokens x 4 heads).
 *  - Every call looks up the array's device address (cudaGetSymbolAddress) on the calling
 *    thread's current device, so a device reset in between is harmless.  The first call on a
 *    device also sets the device up (and may load the library's device code): make that first
 *    call before any stream capture.  It allocates nothing: no cudaMalloc, no cudaFree, no
 *    allocating library routine.
 *  - Every call shares the one array, which keeps the previous call's contents (nothing in it
 *    needs to start at zero).  Calls that may overlap on the GPU -- on different streams, or from
 *    several host threads -- race on it; serialise them on one stream.
 *  - Device status (malformed cu_seqlens) is not readable through kda_read_device_status, which
 *    needs the workspace pointer; the outputs are then left unwritten. */
#define KDA_STATIC_WS_BYTES ((size_t)64 << 20)
kda_status kda_fwd_static_ws(const kda_problem* p, const void* q, const void* k, const void* v,
                             const void* beta, const float* g_or_a, const float* A_log,
                             const float* dt_bias, const float* h0, void* o, float* ht,
                             kda_stream_t stream);

/* Backward of L = sum(o * dO) + sum(ht * dht) for the same inputs as kda_fwd.
 * saved: the set written by kda_fwd for exactly these inputs, or NULL to recompute the forward
 * (checkpoint replay).  dht nullable (zero).  Outputs: dq, dk, dv [T,H,128] and dbeta [T,H]
 * (fp32 or bf16 per out_fp32); dg_or_da fp32 [T,H,128] = dL/dg in g form, dL/da in raw form; in raw form also dA_log
 * fp32 [H] and ddt_bias fp32 [H,128] (ignored, may be NULL, in g form); dh0 fp32
 * [N,H,128,128] nullable.  Source: the chunked KDA training package page (PR #8909), summary
 * (backward path saved / replay) and first commit message (gate gradient dg, dA_log, dt_bias). */
kda_status kda_bwd(const kda_problem* p, const void* q, const void* k, const void* v,
                   const void* beta, const float* g_or_a, const float* A_log,
                   const float* dt_bias, const float* h0, const void* dO, const float* dht,
                   const void* saved, void* dq, void* dk, void* dv, void* dbeta, float* dg_or_da,
                   float* dA_log, float* ddt_bias, float* dh0, void* ws, size_t ws_bytes,
                   kda_stream_t stream);

/* Fragment summaries: `p` describes fragments as documents (p->cu_seqlens = fragment offsets,
 * p->N = number of fragments F).  Each fragment starts its own chunking.
 *   mode KDA_FRAG_FWD: M fp32 [F,H,128,128] = product over the fragment's tokens (later on the
 *     left) of (I - beta k k^T) Diag(exp g);  B_or_C fp32 [F,H,128,128] = the fragment's final
 *     state from S = 0.  Then the fragment maps S_in to S_out = M S_in + B.  dO unused.
 *   mode KDA_FRAG_BWD: B_or_C = C, the gradient at the fragment's first state of sum(o * dO) with
 *     zero end gradient.  M unused (may be NULL).
 * Source: the KCP transfer-walk page (PR #7176), PR description: FP32 affine state summaries,
 * S_out = M * S_in + B, M, B and the states stored in FP32. */
kda_status kda_fragment_summary(const kda_problem* p, int mode, const void* q, const void* k,
                                const void* v, const void* beta, const float* g_or_a,
                                const float* A_log, const float* dt_bias, const void* dO,
                                float* M, float* B_or_C, void* ws, size_t ws_bytes,
                                kda_stream_t stream);

/* Product format of the transfer walk.  M, B (or C) and the states stay FP32 in memory; each
 * format differs only in how the FP32 products M S are formed:
 *   KDA_WALK_FP32       CUDA-core FP32 multiply-add (one block per 32 state columns).
 *   KDA_WALK_TF32       tensor cores (tcgen05 kind::tf32), operands rounded to TF32 (11
 *                       significant bits), one product; full width (one block per document-head).
 *   KDA_WALK_TF32_HILO  tensor cores, each operand split into a TF32 hi and lo part, three
 *                       products (hi hi + hi lo + lo hi); full width.
 *   KDA_WALK_BF16X3     tensor cores (kind::f16), each operand split into three bf16 parts, the
 *                       six part products of combined order < 3; full width.
 *   KDA_WALK_BF16X3_HW  as KDA_WALK_BF16X3, half width: two blocks per (document, head), each
 *                       covering 64 of the state's 128 columns.
 * Source: the KCP transfer-walk page (flashinfer PR #7176), PR description (the shipped walk uses
 * three bf16 pieces per FP32 operand on the tensor cores, FP32 accumulation, two CTAs per
 * (segment, head); the full-width TF32 hi/lo walk it replaced) and the commit note that lists the
 * TF32 hi/lo, static precision-mode and full-width BF16x3 forms. */
typedef enum kda_walk_precision {
    KDA_WALK_FP32 = 0,
    KDA_WALK_TF32 = 1,
    KDA_WALK_TF32_HILO = 2,
    KDA_WALK_BF16X3 = 3,
    KDA_WALK_BF16X3_HW = 4
} kda_walk_precision;

/* Transfer walk over the fragments of N documents.  doc_frag: device int32 [N+1]; the fragments
 * of document n are doc_frag[n] .. doc_frag[n+1]-1 (in token order) and doc_frag[N] = F.
 *   reverse = 0:  S_in[first] = S0[n] (NULL: zero);  S_in[f+1] = M_f S_in[f] + B_f;
 *                 S_final[n] = M_last S_in[last] + B_last  (the document's final state).
 *   reverse = 1 (backward; pass C as B and the documents' dht as S0):
 *                 dS_end[last] = S0[n];  dS_end[f-1] = M_f^T dS_end[f] + C_f;
 *                 S_final[n] = M_first^T dS_end[first] + C_first  (the document's dh0).
 * S_in fp32 [F,H,128,128] receives S_in[f] (forward) or dS_end[f] (backward); S_final fp32
 * [N,H,128,128] nullable.  precision: a kda_walk_precision (all but KDA_WALK_TF32 are accurate
 * to FP32 rounding).  Needs no workspace; `ws` (nullable, >= 256 bytes, 16-byte aligned) only
 * receives a device-side status in its first word (KDA_ERR_TIMEOUT if a bounded wait of the
 * tensor-core walk gave up, S_in / S_final then unspecified), read with kda_read_device_status.
 * Source: the KCP transfer-walk page (PR #7176), PR description (the walk carries the FP32 state
 * across fragment boundaries as S_out = M * S_in + B). */
kda_status kda_transfer_walk(int32_t N, const int32_t* doc_frag, int32_t F, int32_t H,
                             const float* M, const float* B, const float* S0, int reverse,
                             int precision, float* S_in, float* S_final, void* ws,
                             kda_stream_t stream);

/* Width-4 causal depthwise conv1d + SiLU, the step ahead of KDA's q, k and v.  Per document of
 * the pack (cu_seqlens) and channel c:
 *     z[t, c] = bias[c] + sum_{j=0..3} w[c, j] * x[t - 3 + j, c],    y[t, c] = silu(z[t, c])
 * (activation = 0: y = z).  A read before a document's first token takes the document's halo
 * row -- halo[n, 3 + (t - 3 + j - start), c], the three tokens that precede the document, e.g.
 * the end of the previous fragment of the same long document -- or zero when halo is NULL.
 * Layouts: x, halo bf16 [T, C] and [N, 3, C]; w fp32 [C, 4] (tap j multiplies x[t - 3 + j]);
 * bias fp32 [C] (nullable); y, dy, dx and dhalo are fp32 when out_fp32 = 1, else bf16; dw fp32
 * [C, 4], dbias fp32 [C].  C is a multiple of 8 (q, k or v of H heads: C = 128 H; or the three
 * together).  cu_seqlens as for kda_fwd (a malformed one gives unspecified values, never an
 * out-of-bounds access).  The backward (of L = sum(y * dy)) recomputes z, needs the workspace of
 * kda_conv_workspace_size (partial sums of dw and dbias, reduced in a fixed order: results are
 * bitwise reproducible) and writes dhalo (nullable; requires halo) with the gradient flowing into
 * the halo rows.  Source: the KCP transfer-walk page (flashinfer PR #7176), PR description: the
 * module forward runs the conv halo exchange and the conv ahead of the KDA recurrence, and the
 * family ships a width-4 causal conv1d + SiLU training backend with a halo variant. */
typedef struct kda_conv_problem {
    int64_t T;                  /* tokens, >= 0 */
    int32_t N;                  /* documents (or fragments), >= 1 */
    int32_t C;                  /* channels, a positive multiple of 8 */
    int32_t activation;         /* 1: SiLU; 0: none */
    int32_t out_fp32;           /* 1: y, dy, dx, dhalo fp32; 0: bf16 */
    const int32_t* cu_seqlens;  /* device int32 [N+1] */
} kda_conv_problem;
kda_status kda_conv_workspace_size(const kda_conv_problem* p, size_t* ws_bytes);
kda_status kda_conv_fwd(const kda_conv_problem* p, const void* x, const float* w,
                        const float* bias, const void* halo, void* y, kda_stream_t stream);
kda_status kda_conv_bwd(const kda_conv_problem* p, const void* x, const float* w,
                        const float* bias, const void* halo, const void* dy, void* dx, float* dw,
                        float* dbias, void* dhalo, void* ws, size_t ws_bytes, kda_stream_t stream);

/* Copies the device status word of `ws` to the host (synchronises `stream`) and clears it.
 * *device_status receives a kda_status value (KDA_OK when no device-side error happened). */
kda_status kda_read_device_status(void* ws, int* device_status, kda_stream_t stream);

/* Diagnostic (the pages have no counterpart): launches one kernel whose bounded device-side wait
 * cannot complete (an mbarrier nothing arrives on).  After limit_us microseconds of GPU global
 * time (1 .. 1,000,000) the wait gives up and the kernel writes KDA_ERR_TIMEOUT into the status
 * word at the start of `ws` and returns, exactly as the library's kernels report a timed-out
 * wait; the context stays usable.  ws: >= 256 bytes of 16-byte aligned device memory (any
 * workspace), read with kda_read_device_status.  Returns KDA_ERR_INVALID_ARG for a null or
 * misaligned ws or a limit out of range; does not synchronise `stream`. */
kda_status kda_selftest_wait_timeout(void* ws, uint32_t limit_us, kda_stream_t stream);

/* Instrumentation (no effect on results).  Every kernel launch is counted; while profiling is
 * enabled each launch is also bracketed by CUDA events recorded on its stream.
 * kda_profile_collect waits for the recorded events and returns, per kernel kind (index <
 * kda_kernel_count()), the summed device milliseconds and launch counts since the last collect;
 * either array may be NULL. */
kda_status kda_profile_enable(int enable);
kda_status kda_profile_collect(double* ms_per_kind, uint64_t* launches_per_kind);
int kda_kernel_count(void);
const char* kda_kernel_name(int kind);
uint64_t kda_launch_counter(void);

/* Human-readable text of a status; never NULL. */
const char* kda_status_string(kda_status s);

#ifdef __cplusplus
}
#endif

#endif /* KDA_GB300_H */
