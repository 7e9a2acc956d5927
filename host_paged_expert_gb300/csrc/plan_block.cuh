// The device LRU planner as a block-level function, shared by the standalone
// planner kernel and the one-kernel decode step, so both make the same plan.
//
// "Paged Experts" (SGLang docs), "A step: waves, page-in, merge", steps 1-3,
// and "Captured decode": the LRU decision is made on the GPU and written as a
// page-in plan (experts, slots, count) to device buffers.
//
// Conventions the CPU reference fixes and the planner reproduces bit for bit:
//   routing: top-k by logit, ties to the lower expert id, NaN as -inf;
//   D = distinct routed ids; order = resident members of D (ascending id)
//   followed by the others (ascending id), cut into waves of K;
//   per wave: clock += 1; resident members get tick = clock; victims are the
//   slots whose expert is outside the wave, by (tick, slot) ascending; the
//   missing members in ascending id take the victims in that order and get
//   tick = clock.
//
// The planner sits on the critical path of every decode step, so it is
// written for latency: all of its global loads are issued up front, routing
// works on logits held in registers with warp reductions, and everything after
// routing runs in shared memory until the final stores.
#pragma once

#include <math.h>

#include "pe_device.cuh"
#include "pe_internal.h"

namespace pe {

// Order-preserving 32-bit key of a logit (larger logit -> larger key); -0 and
// +0 share a key, as they compare equal.
__device__ __forceinline__ uint32_t logit_key(float v) {
    if (v == 0.f) v = 0.f;
    const uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// One warp routes one token: top-k ids in selection order and the softmax
// over the chosen logits (equal to the E-wide softmax renormalised on them).
// EPL = logits per lane (ceil(E / 32)), held in registers.  Each of the k
// picks takes the lane-local best candidate strictly after the previous pick
// (larger logit first, then lower id), a warp max-reduction of its key, and a
// min-reduction of the ids that carry that key.  Lane j < k returns pick j in
// (id, w); other lanes return id = -1.
template <int EPL>
__device__ __forceinline__ void route_token_warp(const float* __restrict__ row, int E, int k, int& out_id,
                                                 float& out_w, bool& nan_seen) {
    const int lane = threadIdx.x & 31;
    float v[EPL];
    uint32_t key[EPL];
#pragma unroll
    for (int q = 0; q < EPL; ++q) {
        const int e = lane + 32 * q;
        float x = e < E ? row[e] : -INFINITY;
        if (isnan(x)) {
            x = -INFINITY;
            nan_seen = true;
        }
        v[q] = x;
        key[q] = logit_key(x);
    }
    uint32_t prev_key = 0xffffffffu;
    int prev_id = -1;
    float my_v = -INFINITY;
    int my_id = -1;
    for (int j = 0; j < k; ++j) {
        uint32_t bk = 0;
        int bid = 0x7fffffff;
        bool have = false;
#pragma unroll
        for (int q = 0; q < EPL; ++q) {
            const int e = lane + 32 * q;
            // only experts that exist and come strictly after the previous pick
            const bool after = j == 0 || key[q] < prev_key || (key[q] == prev_key && e > prev_id);
            if (e < E && after && (!have || key[q] > bk)) {  // ids ascend with q: first wins a tie
                bk = key[q];
                bid = e;
                have = true;
            }
        }
        const uint32_t mk = __reduce_max_sync(0xffffffffu, have ? bk : 0u);
        const uint32_t cand = (have && bk == mk) ? (uint32_t)bid : 0xffffffffu;
        const int mid = (int)__reduce_min_sync(0xffffffffu, cand);
        if (lane == j) my_id = mid;
        prev_key = mk;
        prev_id = mid;
    }
    // the chosen logits: lane j fetches the value of pick j from its owner lane
#pragma unroll
    for (int q = 0; q < EPL; ++q) {
        const int owner_q = (my_id >= 0) ? (my_id >> 5) : 0;
        const float cand_v = __shfl_sync(0xffffffffu, v[q], (my_id >= 0 ? my_id : 0) & 31);
        if (lane < k && owner_q == q) my_v = cand_v;
    }
    const float v0 = __shfl_sync(0xffffffffu, my_v, 0);
    float ex = 0.f;
    if (lane < k) ex = (v0 == -INFINITY) ? 1.f : expf(my_v - v0);
    float sum = ex;
#pragma unroll
    for (int o = 16; o; o >>= 1) sum = __fadd_rn(sum, __shfl_xor_sync(0xffffffffu, sum, o));
    out_id = lane < k ? my_id : -1;
    out_w = lane < k ? __fdiv_rn(ex, sum) : 0.f;
}

// Routed ids of entries i0, i0 + stride, ... (kPlanBatch of them, kNoEntry
// past nent), all loads issued before any is used.
constexpr int kPlanBatch = 8;
constexpr int kNoEntry = -0x7fffffff;
__device__ __forceinline__ void load_ids(const int32_t* ids, int i0, int stride, int nent, int (&id)[kPlanBatch]) {
#pragma unroll
    for (int u = 0; u < kPlanBatch; ++u) {
        const int i = i0 + u * stride;
        id[u] = i < nent ? ids[i] : kNoEntry;
    }
}

// Where each CTA that plans a single-wave step side by side with others keeps
// the plan (shared memory of the caller).
struct PlanOut {
    int32_t* mexp;  // [K] members: the page-ins in plan order, then the hits
    int32_t* mslot; // [K] their slots
    int32_t* ekey;  // [T*k] slot of each entry, -1 if its expert is not in the wave
    float* ew;      // [T*k] router weight of each entry
    int* count;     // page-ins
    int* size;      // members
};

// One CTA plans every wave of a step (every thread of the block calls this).
// With read_ctr set, `readers` CTAs plan the same step side by side (from the
// same inputs, so to the same plan), each keeping wave 0 in `out`; each counts
// itself in *read_ctr once it holds the old LRU state in shared memory, and
// the CTA that counts last - when no CTA still reads the old state - writes
// the routing, the plan, the new state and the counters to global memory.
// That needs the routed ids in shared memory (T * k <= CAP).  Without
// read_ctr the calling CTA alone plans and writes everything.
// blockDim.x is a multiple of 32 and at least E (thread e owns expert e in the
// scans) and K (thread s owns slot s); CAP >= max(E, K) sizes the shared
// arrays, and an inline-routed step keeps its ids in shared memory when
// T * k <= CAP.  EPL = ceil(E / 32) logits per lane.
template <int EPL, int CAP>
__device__ void plan_block(const LayerDev& L, const Shape& s, const float* logits, int T, int route_inline,
                           uint32_t* err, const PlanOut* out = nullptr, unsigned* read_ctr = nullptr,
                           unsigned readers = 0) {
    __shared__ int32_t sh_slot_expert[CAP];
    __shared__ uint32_t sh_tick[CAP];
    __shared__ int32_t sh_expert_slot[CAP];
    __shared__ int32_t sh_order[CAP];
    __shared__ int32_t sh_wave_of[CAP];
    __shared__ int32_t sh_slot_in_wave[CAP];
    __shared__ int32_t sh_ids[CAP];  // routed ids of an inline-routed step (T*k <= CAP)
    __shared__ uint8_t sh_used[CAP];
    __shared__ uint8_t sh_inwave[CAP];
    __shared__ uint8_t sh_loaded[CAP];
    __shared__ unsigned long long sh_vkey[CAP];  // (tick, slot) of victim slots, ~0 otherwise
    __shared__ int sh_wr[32], sh_wm[32];
    __shared__ int sh_nR, sh_nM, sh_cold, sh_bad, sh_nan, sh_pub;
    __shared__ uint32_t sh_clock;

    const int tid = threadIdx.x, nthr = blockDim.x;
    const int lane = tid & 31, warp = tid >> 5, nwarps = nthr >> 5;
    const int E = s.E, K = s.K, k = s.k;
    const int nent = T * k;
    const bool ids_in_smem = route_inline && nent <= CAP;
    const bool shared_plan = read_ctr != nullptr;

    // The old LRU state is loaded into registers (thread s owns slot s, thread
    // e expert e) and moved to shared memory only after routing: a store of a
    // loaded value waits for its load, so storing first would put one memory
    // round trip per array in front of routing.  This way the state's loads,
    // the logits' loads and the routing overlap.
    int32_t r_slot_expert = -1, r_expert_slot = -1;
    uint32_t r_tick = 0, r_clock = 0;
    uint8_t r_loaded = 0;
    if (tid < K) {
        r_slot_expert = L.slot_expert[tid];
        r_tick = L.slot_tick[tid];
    }
    if (tid < E) {
        r_expert_slot = L.expert_slot[tid];
        r_loaded = L.loaded[tid];
        sh_used[tid] = 0;
        sh_inwave[tid] = 0;
        sh_wave_of[tid] = -1;
        sh_slot_in_wave[tid] = -1;
    }
    if (tid == 0) {
        r_clock = *L.clock;
        sh_cold = 0;
        sh_bad = 0;
        sh_nan = 0;
    }
    if (route_inline) {
        for (int t = warp; t < T; t += nwarps) {
            int id;
            float w;
            bool nan_seen = false;
            route_token_warp<EPL>(logits + (size_t)t * E, E, k, id, w, nan_seen);
            if (lane < k) {
                if (!shared_plan) {
                    L.topk_id[(size_t)t * k + lane] = id;
                    L.topk_w[(size_t)t * k + lane] = w;
                }
                if (ids_in_smem) sh_ids[t * k + lane] = id;
                if (out) out->ew[t * k + lane] = w;
            }
            if (nan_seen) sh_nan = 1;
        }
    }
    if (tid < K) {
        sh_slot_expert[tid] = r_slot_expert;
        sh_tick[tid] = r_tick;
    }
    if (tid < E) {
        sh_expert_slot[tid] = r_expert_slot;
        sh_loaded[tid] = r_loaded;
    }
    if (tid == 0) sh_clock = r_clock;
    __syncthreads();  // routing, state and flags are in shared memory from here on
    // this CTA no longer reads the old state; the last one to say so publishes
    // (the count returned is first used at the end, so nothing waits for it)
    unsigned readers_before = 0;
    if (shared_plan && tid == 0)
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                     : "=r"(readers_before)
                     : "l"(read_ctr)
                     : "memory");
    uint32_t clock = sh_clock;

    for (int i0 = tid; i0 < nent; i0 += kPlanBatch * nthr) {
        int id[kPlanBatch];
        load_ids(ids_in_smem ? sh_ids : L.topk_id, i0, nthr, nent, id);
#pragma unroll
        for (int u = 0; u < kPlanBatch; ++u) {
            const int e = id[u];
            if (e == kNoEntry) continue;
            if (e >= 0 && e < E)
                sh_used[e] = 1;
            else
                sh_bad = 1;
        }
    }
    __syncthreads();

    // order = R ++ M, both ascending id (one scan for both lists)
    const int e = tid;
    const bool used = e < E && sh_used[e];
    const bool isR = used && sh_expert_slot[e] >= 0;
    const bool isM = used && sh_expert_slot[e] < 0;
    const unsigned bR = __ballot_sync(0xffffffffu, isR), bM = __ballot_sync(0xffffffffu, isM);
    const unsigned below = (1u << lane) - 1u;
    if (lane == 0) {
        sh_wr[warp] = __popc(bR);
        sh_wm[warp] = __popc(bM);
    }
    __syncthreads();
    if (warp == 0) {
        const int vr = lane < nwarps ? sh_wr[lane] : 0, vm = lane < nwarps ? sh_wm[lane] : 0;
        int ir = vr, im = vm;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int nr = __shfl_up_sync(0xffffffffu, ir, o), nm = __shfl_up_sync(0xffffffffu, im, o);
            if (lane >= o) {
                ir += nr;
                im += nm;
            }
        }
        if (lane < nwarps) {
            sh_wr[lane] = ir - vr;
            sh_wm[lane] = im - vm;
        }
        if (lane == 31) {
            sh_nR = ir;
            sh_nM = im;
        }
    }
    __syncthreads();
    const int nR = sh_nR, nM = sh_nM;
    if (isR) sh_order[sh_wr[warp] + __popc(bR & below)] = e;
    if (isM) sh_order[nR + sh_wm[warp] + __popc(bM & below)] = e;
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
                if (!shared_plan) {
                    L.member_expert[(size_t)w * K + nmiss + i] = m;
                    L.member_slot[(size_t)w * K + nmiss + i] = slot;
                }
                if (out && w == 0) {
                    out->mexp[nmiss + i] = m;
                    out->mslot[nmiss + i] = slot;
                }
            }
        }
        __syncthreads();
        // rank of each victim slot in (tick, slot) order
        unsigned long long my_key = ~0ull;
        if (tid < K) {
            const int ex = sh_slot_expert[tid];
            if (ex < 0 || !sh_inwave[ex]) my_key = ((unsigned long long)sh_tick[tid] << 32) | (unsigned)tid;
            sh_vkey[tid] = my_key;
        }
        __syncthreads();
        int my_rank = -1;
        if (tid < K && my_key != ~0ull && nmiss > 0) {
            int r = 0;
#pragma unroll 8
            for (int o = 0; o < K; ++o) r += sh_vkey[o] < my_key;
            my_rank = r;
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
            if (!shared_plan) {
                L.plan_expert[q] = m;
                L.plan_slot[q] = slot;
                L.member_expert[q] = m;
                L.member_slot[q] = slot;
                if (!sh_loaded[m]) atomicOr(err, PE_DEVERR_NOT_LOADED);
            }
            if (out && w == 0) {
                out->mexp[my_rank] = m;
                out->mslot[my_rank] = slot;
            }
        }
        __syncthreads();
        for (int i = tid; i < size; i += nthr) {
            const int m = sh_order[base + i];
            sh_wave_of[m] = w;
            sh_slot_in_wave[m] = sh_expert_slot[m];
            sh_inwave[m] = 0;
        }
        if (tid == 0) {
            if (!shared_plan) {
                L.plan_count[w] = nmiss;
                L.member_count[w] = size;
            }
            if (out && w == 0) {
                *out->count = nmiss;
                *out->size = size;
            }
        }
        total_miss += nmiss;
        __syncthreads();
    }
    if (out && nW == 0 && tid == 0) {
        *out->count = 0;
        *out->size = 0;
    }
    if (shared_plan) {  // a single wave (T * k <= K): its plan is in `out`
        if (tid == 0) sh_pub = readers_before == readers - 1;
        __syncthreads();
        if (!sh_pub) {
            for (int i = tid; i < nent; i += nthr) {
                const int m = sh_ids[i];
                out->ekey[i] = m >= 0 && m < E && sh_wave_of[m] == 0 ? sh_slot_in_wave[m] : -1;
            }
            return;
        }
        const int nmiss = *out->count, size = *out->size;
        for (int i = tid; i < size; i += nthr) {
            const int m = out->mexp[i];
            L.member_expert[i] = m;
            L.member_slot[i] = out->mslot[i];
            if (i < nmiss) {
                L.plan_expert[i] = m;
                L.plan_slot[i] = out->mslot[i];
                if (!sh_loaded[m]) atomicOr(err, PE_DEVERR_NOT_LOADED);
            }
        }
        if (tid == 0 && nW > 0) {
            L.plan_count[0] = nmiss;
            L.member_count[0] = size;
        }
    }
    for (int w = nW + tid; w < s.Wmax; w += nthr) {
        L.plan_count[w] = 0;
        L.member_count[w] = 0;
    }

    for (int i0 = tid; i0 < nent; i0 += kPlanBatch * nthr) {
        int id[kPlanBatch];
        load_ids(ids_in_smem ? sh_ids : L.topk_id, i0, nthr, nent, id);
#pragma unroll
        for (int u = 0; u < kPlanBatch; ++u) {
            const int m = id[u], i = i0 + u * nthr;
            if (m == kNoEntry) continue;
            const bool ok = m >= 0 && m < E;
            L.entry_wave[i] = ok ? sh_wave_of[m] : -1;
            L.entry_slot[i] = ok ? sh_slot_in_wave[m] : 0;
            if (shared_plan) {
                L.topk_id[i] = m;
                L.topk_w[i] = out->ew[i];
            }
            if (out) out->ekey[i] = ok && sh_wave_of[m] == 0 ? sh_slot_in_wave[m] : -1;
        }
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
        if (sh_nan) atomicOr(err, PE_DEVERR_NAN_LOGIT);
    }
}

}  // namespace pe
