// Routing and LRU wave planning on the device.
//
// "Paged Experts" (SGLang docs), "A step: waves, page-in, merge", steps 1-3,
// and "Captured decode": the LRU decision is made on the GPU and written as a
// page-in plan (experts, slots, count) to device buffers, so a step needs no
// host synchronisation.  This kernel plans every wave of a step, not only the
// single decode wave, so prefill is planned on the device too.
//
// Conventions the CPU reference fixes and this kernel reproduces bit for bit:
//   routing: top-k by logit, ties to the lower expert id, NaN as -inf;
//   D = distinct routed ids; order = resident members of D (ascending id)
//   followed by the others (ascending id), cut into waves of K;
//   per wave: clock += 1; resident members get tick = clock; victims are the
//   slots whose expert is outside the wave, by (tick, slot) ascending; the
//   missing members in ascending id take the victims in that order and get
//   tick = clock.

#include <math.h>

#include "pe_internal.h"

namespace pe {
namespace {

// Selection order: larger logit first, equal logits -> lower id first.
__device__ __forceinline__ bool ranks_before(float v, int id, float bv, int bid) {
    return v > bv || (v == bv && id < bid);
}

// One warp routes one token: top-k ids in selection order and the softmax
// over the chosen logits (equal to the E-wide softmax renormalised on them).
__device__ void route_token_warp(const float* __restrict__ row, int E, int k, int32_t* ids,
                                 float* ws, uint32_t* err) {
    const int lane = threadIdx.x & 31;
    float prev_v = 0.f;
    int prev_id = -1;
    float my_v = -INFINITY;
    int my_id = 0;
    bool nan_seen = false;
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int bid = 0x7fffffff;
        for (int e = lane; e < E; e += 32) {
            float v = row[e];
            if (isnan(v)) {
                v = -INFINITY;
                nan_seen = true;
            }
            // only candidates strictly after the previous pick qualify
            const bool after = (j == 0) || ranks_before(prev_v, prev_id, v, e);
            if (after && ranks_before(v, e, bv, bid)) {
                bv = v;
                bid = e;
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oid = __shfl_xor_sync(0xffffffffu, bid, o);
            if (ranks_before(ov, oid, bv, bid)) {
                bv = ov;
                bid = oid;
            }
        }
        if (lane == j) {
            my_v = bv;
            my_id = bid;
        }
        prev_v = bv;
        prev_id = bid;
    }
    const float v0 = __shfl_sync(0xffffffffu, my_v, 0);
    float ex = 0.f;
    if (lane < k) ex = (v0 == -INFINITY) ? 1.f : expf(my_v - v0);
    float sum = ex;
#pragma unroll
    for (int o = 16; o; o >>= 1) sum = __fadd_rn(sum, __shfl_xor_sync(0xffffffffu, sum, o));
    if (lane < k) {
        ids[lane] = my_id;
        ws[lane] = __fdiv_rn(ex, sum);
    }
    if (__any_sync(0xffffffffu, nan_seen) && lane == 0) atomicOr(err, PE_DEVERR_NAN_LOGIT);
}

__global__ void __launch_bounds__(256) route_kernel(LayerDev L, int E, int k, const float* logits,
                                                    int T, uint32_t* err) {
    const int warp = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (warp >= T) return;
    route_token_warp(logits + (size_t)warp * E, E, k, L.topk_id + (size_t)warp * k,
                     L.topk_w + (size_t)warp * k, err);
}

// Exclusive block-wide prefix count of a per-thread flag; every thread of the
// block calls it.  warp_tot needs 32 ints.
__device__ __forceinline__ int block_prefix(bool flag, int* warp_tot, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const unsigned b = __ballot_sync(0xffffffffu, flag);
    const int in_warp = __popc(b & ((1u << lane) - 1u));
    if (lane == 0) warp_tot[warp] = __popc(b);
    __syncthreads();
    if (warp == 0) {
        const int v = lane < nwarps ? warp_tot[lane] : 0;
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += n;
        }
        if (lane < nwarps) warp_tot[lane] = incl - v;
        if (lane == 31) *total = incl;
    }
    __syncthreads();
    const int r = warp_tot[warp] + in_warp;
    __syncthreads();
    return r;
}

// One CTA plans every wave of a step.  blockDim.x is a multiple of 32 and at
// least E (thread e owns expert e in the scans) and K (thread s owns slot s).
__global__ void __launch_bounds__(kPlanMaxThreads) plan_kernel(LayerDev L, Shape s,
                                                               const float* logits, int T,
                                                               int route_inline, uint32_t* err) {
    __shared__ int32_t sh_slot_expert[kMaxSlots];
    __shared__ uint32_t sh_tick[kMaxSlots];
    __shared__ int32_t sh_expert_slot[kMaxExperts];
    __shared__ int32_t sh_order[kMaxExperts];
    __shared__ int32_t sh_wave_of[kMaxExperts];
    __shared__ int32_t sh_slot_in_wave[kMaxExperts];
    __shared__ int32_t sh_ids[kMaxExperts];  // routed ids of an inline-routed step (T*k <= 1024)
    __shared__ uint8_t sh_used[kMaxExperts];
    __shared__ uint8_t sh_inwave[kMaxExperts];
    __shared__ int sh_warp[32];
    __shared__ int sh_nR, sh_nM, sh_cold, sh_bad;

    const int tid = threadIdx.x, nthr = blockDim.x;
    const int E = s.E, K = s.K, k = s.k;
    const int nent = T * k;
    const bool ids_in_smem = route_inline && nent <= kMaxExperts;

    // state loads first: they do not depend on routing
    for (int i = tid; i < K; i += nthr) {
        sh_slot_expert[i] = L.slot_expert[i];
        sh_tick[i] = L.slot_tick[i];
    }
    for (int e = tid; e < E; e += nthr) {
        sh_expert_slot[e] = L.expert_slot[e];
        sh_used[e] = 0;
        sh_inwave[e] = 0;
        sh_wave_of[e] = -1;
        sh_slot_in_wave[e] = -1;
    }
    if (tid == 0) {
        sh_cold = 0;
        sh_bad = 0;
    }
    uint32_t clock = *L.clock;
    if (route_inline) {
        for (int t = tid >> 5; t < T; t += nthr >> 5) {
            route_token_warp(logits + (size_t)t * E, E, k, L.topk_id + (size_t)t * k,
                             L.topk_w + (size_t)t * k, err);
            if (ids_in_smem && (tid & 31) < k) sh_ids[t * k + (tid & 31)] = L.topk_id[(size_t)t * k + (tid & 31)];
        }
    }
    __syncthreads();  // publishes the routing (shared and global) to the block

    for (int i = tid; i < nent; i += nthr) {
        const int e = ids_in_smem ? sh_ids[i] : L.topk_id[i];
        if (e >= 0 && e < E)
            sh_used[e] = 1;
        else
            sh_bad = 1;
    }
    __syncthreads();

    // order = R ++ M, both ascending id
    const int e = tid;
    const bool used = e < E && sh_used[e];
    const bool isR = used && sh_expert_slot[e] >= 0;
    const bool isM = used && sh_expert_slot[e] < 0;
    const int posR = block_prefix(isR, sh_warp, &sh_nR);
    const int posM = block_prefix(isM, sh_warp, &sh_nM);
    const int nR = sh_nR, nM = sh_nM;
    if (isR) sh_order[posR] = e;
    if (isM) sh_order[nR + posM] = e;
    __syncthreads();

    const int nD = nR + nM;
    int nW = (nD + K - 1) / K;
    if (nW > s.Wmax) {  // cannot happen for a consistent Wmax; never overrun the plan arrays
        if (tid == 0) atomicOr(err, PE_DEVERR_PLAN);
        nW = s.Wmax;
    }
    int total_miss = 0;
    for (int w = 0; w < nW; ++w) {
        const int base = w * K;
        const int size = min(K, nD - base);
        const int nres = (w == 0) ? nR : 0;  // only R can be resident, and R fits in wave 0
        const int nmiss = size - nres;
        ++clock;
        for (int i = tid; i < size; i += nthr) {
            const int m = sh_order[base + i];
            sh_inwave[m] = 1;
            if (i < nres) {
                const int slot = sh_expert_slot[m];
                sh_tick[slot] = clock;
                // hits follow the page-ins in the member list
                L.member_expert[(size_t)w * K + nmiss + i] = m;
                L.member_slot[(size_t)w * K + nmiss + i] = slot;
            }
        }
        __syncthreads();
        // rank of each victim slot in (tick, slot) order
        int my_rank = -1;
        if (tid < K) {
            const int ex = sh_slot_expert[tid];
            if (ex < 0 || !sh_inwave[ex]) {
                const unsigned long long key = ((unsigned long long)sh_tick[tid] << 32) | (unsigned)tid;
                int r = 0;
                for (int o = 0; o < K; ++o) {
                    const int ox = sh_slot_expert[o];
                    if (ox < 0 || !sh_inwave[ox]) {
                        const unsigned long long ok = ((unsigned long long)sh_tick[o] << 32) | (unsigned)o;
                        r += ok < key;
                    }
                }
                my_rank = r;
            }
        }
        __syncthreads();
        if (my_rank >= 0 && my_rank < nmiss) {
            const int slot = tid;
            const int m = sh_order[base + nres + my_rank];
            const int old = sh_slot_expert[slot];
            if (old >= 0)
                sh_expert_slot[old] = -1;
            else
                atomicAdd(&sh_cold, 1);
            sh_slot_expert[slot] = m;
            sh_expert_slot[m] = slot;
            sh_tick[slot] = clock;
            const size_t q = (size_t)w * K + my_rank;
            L.plan_expert[q] = m;
            L.plan_slot[q] = slot;
            L.member_expert[q] = m;
            L.member_slot[q] = slot;
            if (!L.loaded[m]) atomicOr(err, PE_DEVERR_NOT_LOADED);
        }
        __syncthreads();
        for (int i = tid; i < size; i += nthr) {
            const int m = sh_order[base + i];
            sh_wave_of[m] = w;
            sh_slot_in_wave[m] = sh_expert_slot[m];
            sh_inwave[m] = 0;
        }
        if (tid == 0) {
            L.plan_count[w] = nmiss;
            L.member_count[w] = size;
        }
        total_miss += nmiss;
        __syncthreads();
    }
    for (int w = nW + tid; w < s.Wmax; w += nthr) {
        L.plan_count[w] = 0;
        L.member_count[w] = 0;
    }

    for (int i = tid; i < nent; i += nthr) {
        const int m = ids_in_smem ? sh_ids[i] : L.topk_id[i];
        const bool ok = m >= 0 && m < E;
        L.entry_wave[i] = ok ? sh_wave_of[m] : -1;
        L.entry_slot[i] = ok ? sh_slot_in_wave[m] : 0;
    }
    for (int i = tid; i < K; i += nthr) {
        L.slot_expert[i] = sh_slot_expert[i];
        L.slot_tick[i] = sh_tick[i];
    }
    for (int m = tid; m < E; m += nthr) L.expert_slot[m] = sh_expert_slot[m];
    if (tid == 0) {
        *L.clock = clock;
        *L.num_waves = nW;
        atomicAdd(&L.counters[C_STEPS], 1ull);
        atomicAdd(&L.counters[C_WAVES], (unsigned long long)nW);
        atomicAdd(&L.counters[C_ENTRIES], (unsigned long long)nent);
        atomicAdd(&L.counters[C_DISTINCT], (unsigned long long)nD);
        atomicAdd(&L.counters[C_HITS], (unsigned long long)nR);
        atomicAdd(&L.counters[C_PAGE_INS], (unsigned long long)total_miss);
        atomicAdd(&L.counters[C_COLD], (unsigned long long)sh_cold);
        if (sh_bad) atomicOr(err, PE_DEVERR_PLAN);
    }
}

}  // namespace

cudaError_t launch_route(const LayerDev& L, const Shape& s, const float* logits, int T,
                         uint32_t* err, cudaStream_t st) {
    const int warps = 8;
    route_kernel<<<(T + warps - 1) / warps, warps * 32, 0, st>>>(L, s.E, s.k, logits, T, err);
    return cudaGetLastError();
}

cudaError_t launch_plan(const LayerDev& L, const Shape& s, const float* logits, int T,
                        int route_inline, uint32_t* err, cudaStream_t st) {
    int threads = s.E > s.K ? s.E : s.K;
    if (route_inline && threads < 32 * T) threads = 32 * T;  // one warp per token
    threads = (threads + 31) / 32 * 32;
    if (threads > kPlanMaxThreads) threads = kPlanMaxThreads;
    plan_kernel<<<1, threads, 0, st>>>(L, s, logits, T, route_inline, err);
    return cudaGetLastError();
}

}  // namespace pe
