// Launch accounting and optional per-kernel CUDA-event timing (instrumentation only).
#include <atomic>
#include <mutex>
#include <vector>

#include "kda_internal.cuh"

namespace kda {

namespace {
std::atomic<uint64_t> g_launches{0};
std::atomic<bool> g_enabled{false};
std::mutex g_mu;
struct Rec {
    int kind;
    cudaEvent_t a, b;
};
std::vector<Rec> g_recs;
const char* const kNames[KK_COUNT] = {"k_plan",      "k_intra_fwd",    "k_chain_fwd",
                                      "k_chain_bwd",    "k_bwd_gemms_tc",    "k_bwd_intra",
                                      "k_param_reduce", "k_walk",         "k_conv_fwd",
                                      "k_conv_bwd",     "k_conv_reduce"};
}  // namespace

const char* kernel_name(int kind) { return (kind >= 0 && kind < KK_COUNT) ? kNames[kind] : "?"; }

ProfScope::ProfScope(int kind, cudaStream_t st) : kind_(kind), st_(st), a_(nullptr), b_(nullptr) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (g_enabled.load(std::memory_order_relaxed) && cudaEventCreate(&a_) == cudaSuccess &&
        cudaEventCreate(&b_) == cudaSuccess)
        cudaEventRecord(a_, st_);
}

ProfScope::~ProfScope() {
    if (!b_) return;
    cudaEventRecord(b_, st_);
    std::lock_guard<std::mutex> lk(g_mu);
    g_recs.push_back({kind_, a_, b_});
}

}  // namespace kda

using namespace kda;

extern "C" {

kda_status kda_profile_enable(int enable) {
    g_enabled.store(enable != 0);
    return KDA_OK;
}

kda_status kda_profile_collect(double* ms_per_kind, uint64_t* launches_per_kind) {
    std::vector<Rec> recs;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        recs.swap(g_recs);
    }
    for (int i = 0; i < KK_COUNT; ++i) {
        if (ms_per_kind) ms_per_kind[i] = 0.0;
        if (launches_per_kind) launches_per_kind[i] = 0;
    }
    kda_status st = KDA_OK;
    for (auto& r : recs) {
        float ms = 0.f;
        if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess)
            st = KDA_ERR_CUDA;
        if (ms_per_kind) ms_per_kind[r.kind] += ms;
        if (launches_per_kind) launches_per_kind[r.kind] += 1;
        cudaEventDestroy(r.a);
        cudaEventDestroy(r.b);
    }
    return st;
}

int kda_kernel_count(void) { return KK_COUNT; }

const char* kda_kernel_name(int kind) { return kernel_name(kind); }

uint64_t kda_launch_counter(void) { return g_launches.load(); }

}  // extern "C"
