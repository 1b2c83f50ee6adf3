// Chunk plan of a call: the chunk table, per-document chunk offsets and the recurrence launch order.
#include "kda_internal.cuh"

namespace kda {

// Builds the chunk table from cu_seqlens on the device (no host synchronisation).  Malformed
// offsets (cu[0] != 0, decreasing, cu[N] != T) set the status word and leave zero chunks, so every
// later kernel of the call does nothing.  One block: each thread counts the chunks of a contiguous
// run of documents, a block-wide exclusive scan gives the runs' first chunks, each thread writes
// its documents' offsets, and each warp writes the chunk-table entries of every NW-th document
// with its 32 lanes (work O(N / threads + chunks / 32) per thread instead of a serial pass).
__global__ void k_plan(Params p) {
    constexpr int NW = NTHR / 32;
    __shared__ long long wtot[NW];
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int per = (p.N + NTHR - 1) / NTHR;
    const int n0 = min(tid * per, p.N), n1 = min(n0 + per, p.N);
    int b = 0;
    long long cnt = 0;  // 64-bit: malformed offsets cannot wrap the sums
    for (int n = n0; n < n1; ++n) {
        const int a = p.cu[n], e = p.cu[n + 1];
        if (e < a) b = 1;
        cnt += (max(e - a, 0) + CH - 1) / CH;
    }
    if (tid == 0) b |= (p.cu[0] != 0) || (int64_t(p.cu[p.N]) != p.T);
    // exclusive scan of cnt over the block
    long long x = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wtot[w] = x;
    __syncthreads();
    long long wbase = 0, total = 0;
    for (int i = 0; i < NW; ++i) {
        if (i < w) wbase += wtot[i];
        total += wtot[i];
    }
    long long acc = wbase + x - cnt;  // first chunk of this thread's documents
    if (total > p.maxC) b = 1;
    for (int n = n0; n < n1; ++n) {
        p.doc_off[n] = int(min(acc, (long long)p.maxC));
        acc += (max(p.cu[n + 1] - p.cu[n], 0) + CH - 1) / CH;
    }
    const int bad = __syncthreads_or(b);
    if (tid == 0) {
        p.doc_off[p.N] = int(min(total, (long long)p.maxC));
        *p.nchunks = bad ? 0 : int(total);
        p.status[0] = bad ? KDA_ERR_DEVICE_CHECK : KDA_OK;  // status of the latest call
    }
    if (bad) {
        __syncthreads();
        for (int n = tid; n <= p.N; n += NTHR) p.doc_off[n] = 0;
        for (int n = tid; n < p.N; n += NTHR) p.doc_order[n] = n;
        return;
    }
    __syncthreads();  // doc_off (global) is written and visible to the block
    // the state recurrences launch their blocks longest document first (ties in index order);
    // above MAX_SORT documents the order stays the identity
    constexpr int MAX_SORT = 1024;
    __shared__ int ncs[MAX_SORT];
    if (p.N > MAX_SORT) {
        for (int i = tid; i < p.N; i += NTHR) p.doc_order[i] = i;
    } else {
        for (int i = tid; i < p.N; i += NTHR) ncs[i] = p.doc_off[i + 1] - p.doc_off[i];
        __syncthreads();
        for (int i = tid; i < p.N; i += NTHR) {
            const int ni = ncs[i];
            int rank = 0;
            for (int j = 0; j < p.N; ++j) rank += (ncs[j] > ni) || (ncs[j] == ni && j < i);
            p.doc_order[rank] = i;
        }
    }
    for (int n = w; n < p.N; n += NW) {
        const int a = p.cu[n], len = p.cu[n + 1] - a, off = p.doc_off[n];
        const int nc = (len + CH - 1) / CH;
        for (int j = lane; j < nc; j += 32) p.chunk_tab[off + j] = make_int4(n, a + CH * j, min(CH, len - CH * j), j);
    }
}

// Group plan of a call with chunk groups (one block, after k_plan): document n's chunks
// [doc_off[n], doc_off[n + 1]) are cut into groups of G chunks (the last one shorter; an empty
// document keeps one empty group, so every document has at least one group and its walk yields
// its final state).  Groups are numbered document by document; unused group slots up to Gmax are
// empty.  The launch order puts longer groups first (ties in index order; above MAX_SORT groups
// the order stays the identity).
__global__ void k_group_plan(Params p, GroupPlan gp) {
    if (threadIdx.x == 0) {
        int g = 0;
        for (int n = 0; n < p.N; ++n) {
            gp.doc_frag[n] = g;
            const int c0 = p.doc_off[n], c1 = p.doc_off[n + 1];
            const int ng = c1 > c0 ? (c1 - c0 + gp.G - 1) / gp.G : 1;
            for (int i = 0; i < ng && g < gp.Gmax; ++i) gp.gdoc_off[g++] = min(c0 + i * gp.G, c1);
        }
        gp.doc_frag[p.N] = g;
        *gp.ngroups = g;
        const int total = p.doc_off[p.N];
        for (int i = g; i <= gp.Gmax; ++i) gp.gdoc_off[i] = total;
    }
    __syncthreads();
    constexpr int MAX_SORT = 1024;
    __shared__ int ncs[MAX_SORT];
    if (gp.Gmax > MAX_SORT) {
        for (int i = threadIdx.x; i < gp.Gmax; i += blockDim.x) gp.gdoc_order[i] = i;
        return;
    }
    for (int i = threadIdx.x; i < gp.Gmax; i += blockDim.x) ncs[i] = gp.gdoc_off[i + 1] - gp.gdoc_off[i];
    __syncthreads();
    for (int i = threadIdx.x; i < gp.Gmax; i += blockDim.x) {
        const int ni = ncs[i];
        int rank = 0;
        for (int j = 0; j < gp.Gmax; ++j) rank += (ncs[j] > ni) || (ncs[j] == ni && j < i);
        gp.gdoc_order[rank] = i;
    }
}

}  // namespace kda
