// Chunk plan of a call: the chunk table, per-document chunk offsets and the recurrence launch order.
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
        for (int n = threadIdx.x; n < p.N; n += blockDim.x) p.doc_order[n] = n;
        return;
    }
    // the state recurrences launch their blocks longest document first (ties in index order);
    // above MAX_SORT documents the order stays the identity
    constexpr int MAX_SORT = 1024;
    __shared__ int ncs[MAX_SORT];
    if (p.N > MAX_SORT) {
        for (int i = threadIdx.x; i < p.N; i += blockDim.x) p.doc_order[i] = i;
    } else {
        for (int i = threadIdx.x; i < p.N; i += blockDim.x) ncs[i] = p.doc_off[i + 1] - p.doc_off[i];
        __syncthreads();
        for (int i = threadIdx.x; i < p.N; i += blockDim.x) {
            const int ni = ncs[i];
            int rank = 0;
            for (int j = 0; j < p.N; ++j) rank += (ncs[j] > ni) || (ncs[j] == ni && j < i);
            p.doc_order[rank] = i;
        }
    }
    for (int n = 0; n < p.N; ++n) {
        const int a = p.cu[n], len = p.cu[n + 1] - a, off = p.doc_off[n];
        const int nc = (len + CH - 1) / CH;
        for (int j = threadIdx.x; j < nc; j += blockDim.x)
            p.chunk_tab[off + j] = make_int4(n, a + CH * j, min(CH, len - CH * j), j);
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
