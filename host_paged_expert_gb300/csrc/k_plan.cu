// Standalone routing and planning kernels (the planner itself is plan_block,
// shared with the one-kernel decode step): route_kernel routes many tokens,
// one warp each, ahead of the planner for prefill-sized steps; plan_kernel
// plans every wave of a step in one CTA, routing inline for small steps.

#include "plan_block.cuh"

namespace pe {
namespace {

template <int EPL>
__global__ void __launch_bounds__(256) route_kernel(LayerDev L, int E, int k, const float* logits,
                                                    int T, uint32_t* err) {
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    int id;
    float w;
    bool nan_seen = false;
    route_token_warp<EPL>(logits + (size_t)t * E, E, k, id, w, nan_seen);
    const int lane = threadIdx.x & 31;
    if (lane < k) {
        L.topk_id[(size_t)t * k + lane] = id;
        L.topk_w[(size_t)t * k + lane] = w;
    }
    if (__any_sync(0xffffffffu, nan_seen) && lane == 0) atomicOr(err, PE_DEVERR_NAN_LOGIT);
}

// One CTA plans every wave of a step (see plan_block).
template <int EPL>
__global__ void __launch_bounds__(kPlanMaxThreads) plan_kernel(LayerDev L, Shape s, const float* logits, int T,
                                                               int route_inline, uint32_t* err) {
    pdl_wait();
    pdl_trigger();
    plan_block<EPL, kMaxExperts>(L, s, logits, T, route_inline, err);
}

inline int epl_for(int E) {
    const int epl = (E + 31) / 32;
    return epl <= 1 ? 1 : epl <= 2 ? 2 : epl <= 4 ? 4 : epl <= 8 ? 8 : epl <= 16 ? 16 : 32;
}

}  // namespace

cudaError_t launch_route(const LayerDev& L, const Shape& s, const float* logits, int T,
                         uint32_t* err, cudaStream_t st) {
    const int warps = 8;
    const int grid = (T + warps - 1) / warps;
    switch (epl_for(s.E)) {
#define PE_ROUTE(N) case N: return launch_pdl(route_kernel<N>, grid, warps * 32, 0, st, L, s.E, s.k, logits, T, err);
        PE_ROUTE(1) PE_ROUTE(2) PE_ROUTE(4) PE_ROUTE(8) PE_ROUTE(16) PE_ROUTE(32)
#undef PE_ROUTE
    }
    return cudaGetLastError();
}

cudaError_t launch_plan(const LayerDev& L, const Shape& s, const float* logits, int T,
                        int route_inline, uint32_t* err, cudaStream_t st) {
    int threads = s.E > s.K ? s.E : s.K;
    if (route_inline && threads < 32 * T) threads = 32 * T;  // one warp per token
    // a large step's entry loops want many threads more than a small barrier
    if ((long long)T * s.k > 4LL * threads) threads = kPlanMaxThreads;
    threads = (threads + 31) / 32 * 32;
    if (threads > kPlanMaxThreads) threads = kPlanMaxThreads;
    switch (epl_for(s.E)) {
#define PE_PLAN(N) case N: return launch_pdl(plan_kernel<N>, 1, threads, 0, st, L, s, logits, T, route_inline, err);
        PE_PLAN(1) PE_PLAN(2) PE_PLAN(4) PE_PLAN(8) PE_PLAN(16) PE_PLAN(32)
#undef PE_PLAN
    }
    return cudaGetLastError();
}

}  // namespace pe
