// A single-wave decode step in one kernel: routing and LRU plan, page-in,
// gate/up, down projection and top-k sum.
//
// "Paged Experts" (SGLang docs), "Captured decode": a decode step whose
// entries fit the K slots (tokens * top_k <= K) is one wave decided and paged
// on the GPU.  Once the plan is written, what bounds that step is the host
// link: the missing experts' bytes must cross it.  This kernel keeps every
// other part of the step underneath that transfer.
//   planner    every CTA routes the tokens and plans the wave itself
//              (plan_block, the same code as the standalone planner), so no
//              CTA waits for a plan to travel through global memory; the
//              last CTA to have read the old LRU state writes the new one;
//   link SMs   stream the page-ins' gate/up rows from the host store (writing
//              them to their slots and computing h from them on the way) and
//              copy the rest of each paged row;
//   HBM SMs    compute h of the resident experts, then - as soon as those are
//              all done - their down projections into the merged buffer;
//   all SMs    once the link is drained: the down projections of the paged
//              experts, then the fixed-order top-k sum.
// A CTA's role follows the SM it runs on (every third SM streams the link):
// outstanding host reads hold an SM's memory pipeline for tens of
// microseconds, and HBM loads issued on the same SM would queue behind them.
// Work inside a role is split statically: every CTA registers its role and
// gets a rank within it while the plan is being made, so no work queue is
// contended during the transfer.  Phases are ordered by
// counters in global memory (bounded waits; the grid is sized so that every
// CTA is resident at once).  The last CTA to leave resets the counters for the
// layer's next step.
//
// Every value is computed by the same device code, in the same order, as in
// the multi-kernel path (row_pair_h for h, the lane-chunked dot product and
// the same tree of additions over the warp for a down row - warp_sum, or
// warp_sum_rows for the 4-bit rows - p = w * d, the sum over j = 0..k-1 from
// zero), so the two paths give the same bits and the output still equals
// K = E.  The down items read the entry's h from a copy in shared memory
// (stage_h), with the same values.

#include "fp4_device.cuh"
#include "fp8_device.cuh"
#include "int4_device.cuh"
#include "pe_device.cuh"
#include "pe_internal.h"
#include "plan_block.cuh"

namespace pe {
namespace {

constexpr int kThr = 256;
constexpr int kWp = kThr / 32;
constexpr int kRowsD = 4;                                 // down rows per warp item
constexpr int kCopyLd = 8;                                // 16-byte loads per lane per copy item
constexpr size_t kCopyItem = (size_t)32 * 16 * kCopyLd;  // 4 KiB
constexpr int kDynBudget = 48 * 1024;
constexpr uint32_t kSpinLimit = 1u << 23;  // polls (>= 128 ns apart): about a second

// Per-layer counters: role registration, completion counts and barriers.
enum SyncSlot { R_LINK = 0, R_HBM, D_LINK, D_HITS, S_DOWN, P_READ, H_TICKET, S_EXIT, S_NUM };
constexpr int kPlanCap = 256;    // planner capacity inside this kernel: E, K <= 256
// CTAs on SMs with %smid % link_every == 0 stream the host link: every third
// SM, or every sixth for int4 steps of two or more tokens.  An int4 page-in is
// a quarter of a bf16 one while the resident experts' GEMVs take about as
// long, and with more tokens those GEMVs are the longer side (measured: at
// batch 4 every sixth SM is 6 % faster than every third, at batch 1 1 %
// slower).
constexpr int kLinkSmEvery = 3, kLinkSmEveryInt4Batch = 6;

// 32-bit words of the per-CTA plan in dynamic shared memory: member experts
// and slots [K each], then entry slot, member index and router weight
// [kFusedMaxEntries each]; staged x follows, 16-byte aligned.
__host__ __device__ __forceinline__ int decode_meta_words(const Shape& s) {
    return (2 * s.K + 3 * kFusedMaxEntries + 3) & ~3;
}
// 32-bit words after the plan that hold one entry's h during the down
// projections (I floats, I a multiple of 8); staged x follows.
__host__ __device__ __forceinline__ int decode_hstage_words(const Shape& s) { return s.I; }

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Bypass L1: data written by other CTAs of this grid.
__device__ __forceinline__ int4 ldcg16(const void* p) { return __ldcg(reinterpret_cast<const int4*>(p)); }

// All threads of the CTA have finished their writes; publish them and count.
__device__ __forceinline__ void cta_arrive(unsigned* ctr) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(ctr, 1u);
    }
}

// Wait (thread 0 polls, the CTA waits at the barrier) until *ctr >= target.
// Gives up after kSpinLimit polls, records PE_DEVERR_TIMEOUT and returns false.
__device__ __forceinline__ bool cta_wait(const unsigned* ctr, unsigned target, uint32_t* err, int* flag_sh,
                                         uint32_t limit = kSpinLimit) {
    if (threadIdx.x == 0) {
        int ok = 0;
        for (uint32_t i = 0; i < limit; ++i) {
            if (ld_acquire_u32(ctr) >= target) {
                ok = 1;
                break;
            }
            __nanosleep(128);
        }
        if (!ok) atomicOr(err, PE_DEVERR_TIMEOUT);
        *flag_sh = ok;
    }
    __syncthreads();
    return *flag_sh != 0;
}

// p = w * (down_m . h) for kRowsD rows m0.. of one entry, written to merged.
// CPL = 16-byte chunks of an I-long row per lane.  h: the entry's h staged in
// shared memory (hs_pos<2> layout).
template <int CPL>
__device__ __forceinline__ void down_rows(const uint8_t* w2, const float* h, float wj, int m0, int H, int I,
                                          float* merged_row, int lane) {
    const int nchunk = I >> 3;
    const size_t row_bytes = (size_t)I * 2;
    int4 wv[kRowsD][CPL];
#pragma unroll
    for (int r = 0; r < kRowsD; ++r)
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            const int idx = lane + 32 * c;
            wv[r][c] = (m0 + r < H && idx < nchunk) ? ldcg16(w2 + (size_t)(m0 + r) * row_bytes + 16 * (size_t)idx)
                                                    : make_int4(0, 0, 0, 0);
        }
    float4 hv[CPL][2];
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
        const int idx = lane + 32 * c;
        if (idx < nchunk) {
            hv[c][0] = reinterpret_cast<const float4*>(h)[hs_pos<2>(idx, 0)];
            hv[c][1] = reinterpret_cast<const float4*>(h)[hs_pos<2>(idx, 1)];
        } else {
            hv[c][0] = hv[c][1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
#pragma unroll
    for (int r = 0; r < kRowsD; ++r) {
        float d = 0.f;
#pragma unroll
        for (int c = 0; c < CPL; ++c)
            if (lane + 32 * c < nchunk) d = dot8_bf16_f32(wv[r][c], hv[c][0], hv[c][1], d);
        d = warp_sum(d);
        if (lane == 0 && m0 + r < H) merged_row[m0 + r] = __fmul_rn(wj, d);
    }
}

// FP8 version: E4M3 codes with the 128x128 block scales of w2 (all kRowsD rows
// lie in one 128-row block), the same arithmetic as the FP8 down kernel; h
// staged in shared memory (hs_pos<4> layout).
template <int CPL>
__device__ __forceinline__ void down_rows_fp8(const uint8_t* w2, const float* s2, const float* h, float wj, int m0,
                                              int H, int I, float* merged_row, int lane) {
    const int nchunk = I >> 4;
    const int nbi = (I + kFp8Block - 1) / kFp8Block;
    const float* srow = s2 + (size_t)(m0 / kFp8Block) * nbi;
    int4 wv[kRowsD][CPL];
#pragma unroll
    for (int r = 0; r < kRowsD; ++r)
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            const int idx = lane + 32 * c;
            wv[r][c] = (m0 + r < H && idx < nchunk) ? ldcg16(w2 + (size_t)(m0 + r) * I + 16 * (size_t)idx)
                                                    : make_int4(0, 0, 0, 0);
        }
    float sc[CPL];
    float4 hv[CPL][4];
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
        const int idx = lane + 32 * c;
        if (idx < nchunk) {
            sc[c] = __ldcg(srow + (idx * 16) / kFp8Block);
#pragma unroll
            for (int v = 0; v < 4; ++v) hv[c][v] = reinterpret_cast<const float4*>(h)[hs_pos<4>(idx, v)];
        } else {
            sc[c] = 0.f;
#pragma unroll
            for (int v = 0; v < 4; ++v) hv[c][v] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
#pragma unroll
    for (int r = 0; r < kRowsD; ++r) {
        float d = 0.f;
#pragma unroll
        for (int c = 0; c < CPL; ++c)
            if (lane + 32 * c < nchunk) d = fmaf(sc[c], dot16_e4m3_f32(wv[r][c], hv[c]), d);
        d = warp_sum(d);
        if (lane == 0 && m0 + r < H) merged_row[m0 + r] = __fmul_rn(wj, d);
    }
}

// Dynamic shared memory: [member experts K][member slots K][entry keys nent]
// [entry member nent] padded to 4 ints, then one entry's h (I floats) for the
// down items, then the tokens' x when it fits.
// Chunks per lane cover H <= 2048 and I <= 1024 (bf16: 8 and 4 chunks of 8
// values, FP8: 4 and 2 chunks of 16 codes, int4: 2 and 1 chunks of 32 codes);
// chunks past the row are skipped, so the arithmetic is that of the exact
// chunk counts.
constexpr int CPLH = 8, CPLI = 4, CPLH8 = 4, CPLI8 = 2, CPLH4 = 2, CPLI4 = 1;
// 4-bit rows are short (H/2 and I/2 bytes), so a resident 4-bit gate/up item
// takes kRowsG4 row pairs and an int4 down item kRowsD4 rows to keep enough
// bytes in flight; the per-row arithmetic is unchanged.
constexpr int kRowsG4 = 2, kRowsD4 = 8, kRowsDFp4 = 4;
// FMT: the expert format (PE_BF16, PE_FP8_BLOCK128, PE_INT4_GPTQ, PE_MXFP4 or
// PE_NVFP4; the three 4-bit formats share the int4 tiling).
template <int EPL, int FMT>
__global__ void __launch_bounds__(kThr, 2) decode_step_kernel(LayerDev L, Shape s, const float* __restrict__ logits,
                                                                  const __nv_bfloat16* __restrict__ x,
                                                                 const uint8_t* __restrict__ host,
                                                                 uint8_t* __restrict__ slots, int T,
                                                                 float* __restrict__ hbuf, float* __restrict__ merged,
                                                                 __nv_bfloat16* __restrict__ out, unsigned* sync,
                                                                 uint32_t* err, int stage_x) {
    extern __shared__ int4 sh_dyn[];
    __shared__ int sh_flag;
    __shared__ int sh_nhit, sh_nmiss;
    __shared__ int sh_hit_list[kFusedMaxEntries], sh_miss_list[kFusedMaxEntries];
    int32_t* sh_mexp = reinterpret_cast<int32_t*>(sh_dyn);
    int32_t* sh_mslot = sh_mexp + s.K;
    int32_t* sh_ekey = sh_mslot + s.K;  // entry's slot (-1 if not in the wave)
    int32_t* sh_eq = sh_ekey + kFusedMaxEntries;  // entry's member index
    float* sh_ew = reinterpret_cast<float*>(sh_eq + kFusedMaxEntries);  // entry's router weight
    __shared__ int sh_count, sh_size;
    const int nent = T * s.k;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    pdl_wait();

    // Every CTA registers the role its SM suggests and gets a rank in it,
    // stages x, and plans the step into its own shared memory.
    __shared__ int sh_link_sm, sh_role_rank;
    if (threadIdx.x == kThr - 32) {  // a warp that routes no token of a small step: it waits for the atomic
        unsigned smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        const unsigned link_every = is_4bit(FMT) && T > 1 ? kLinkSmEveryInt4Batch : kLinkSmEvery;
        sh_link_sm = (smid % link_every) == 0;
        sh_role_rank = (int)atomicAdd(&sync[sh_link_sm ? R_LINK : R_HBM], 1u);
    }
    // x is copied to shared memory asynchronously, underneath the planning
    const uint8_t* xbase = reinterpret_cast<const uint8_t*>(x);
    if (stage_x) {
        int4* sx = reinterpret_cast<int4*>(sh_mexp + decode_meta_words(s) + decode_hstage_words(s));
        const int nvec = T * s.H / 8;
        for (int i = threadIdx.x; i < nvec; i += blockDim.x) {
            const unsigned dst = (unsigned)__cvta_generic_to_shared(sx + i);
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(xbase + 16 * (size_t)i) : "memory");
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
        xbase = reinterpret_cast<const uint8_t*>(sx);
    }
    {
        const PlanOut po{sh_mexp, sh_mslot, sh_ekey, sh_ew, &sh_count, &sh_size};
        plan_block<EPL, kPlanCap>(L, s, logits, T, 1, err, &po, &sync[P_READ], gridDim.x);
    }
    if (stage_x) asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    const int size = sh_size;
    const int count = sh_count;
    if (threadIdx.x < nent) {  // member of each entry (nent <= kFusedMaxEntries <= kThr)
        int q = -1;
        for (int j = 0; j < size; ++j)
            if (sh_mslot[j] == sh_ekey[threadIdx.x]) q = j;
        sh_eq[threadIdx.x] = q;
    }
    __syncthreads();
    if (threadIdx.x == 0) {  // entries of hit members / of paged members, ascending
        int nh = 0, nm = 0;
        for (int i = 0; i < nent; ++i) {
            const int q = sh_eq[i];
            if (q < 0) continue;
            if (q < count)
                sh_miss_list[nm++] = i;
            else
                sh_hit_list[nh++] = i;
        }
        sh_nhit = nh;
        sh_nmiss = nm;
    }
    __syncthreads();

    const int nchunk = s.H >> 3;
    const size_t row_bytes = (size_t)s.H * 2;
    // gate/up row pairs per resident-expert item (a page-in item takes one:
    // the link wants many warps with host reads in flight)
    constexpr int RPI = is_4bit(FMT) ? kRowsG4 : 1;
    constexpr int RD = FMT == PE_INT4_GPTQ ? kRowsD4 : is_4bit(FMT) ? kRowsDFp4 : kRowsD;  // down rows per item
    const int ipe = s.I / RPI;  // gate/up items per resident expert
    const long long miss_rows = (long long)count * s.I;
    const size_t tail_bytes = s.copy_bytes - s.tail_off;
    const long long copies_per = (long long)((tail_bytes + kCopyItem - 1) / kCopyItem);
    const long long link_items = miss_rows + (long long)count * copies_per;
    const long long hbm_items = (long long)(size - count) * ipe;
    const int G = gridDim.x;
    const int row_blocks = (s.H + RD - 1) / RD;
    // roles: registration is complete long before the plan is (bounded wait)
    if (threadIdx.x == 0) {
        bool all = false;
        for (uint32_t i = 0; i < kSpinLimit && !all; ++i) {
            all = ld_acquire_u32(&sync[R_LINK]) + ld_acquire_u32(&sync[R_HBM]) >= (unsigned)G;
            if (!all) __nanosleep(64);
        }
        // CTAs that were not all resident would split the work inconsistently:
        // name the cause here rather than in a later phase wait
        if (!all) atomicOr(err, PE_DEVERR_TIMEOUT);
    }
    __syncthreads();
    const int nL = (int)__ldcg(&sync[R_LINK]), nH = G - nL;
    // split: link SMs stream the page-ins while HBM SMs run the resident experts;
    // with no page-ins, no resident experts, or one group empty, every CTA does both
    const bool split = link_items > 0 && hbm_items > 0 && nL > 0 && nH > 0;
    const bool link_cta = split ? sh_link_sm != 0 : true;
    const bool hbm_cta = split ? sh_link_sm == 0 : true;
    const int rank = split ? sh_role_rank : (int)blockIdx.x;
    const int link_ctas = split ? nL : G, hbm_ctas = split ? nH : G;

    // Gate/up (and page-in) items of one role, strided over that role's CTAs:
    // the link items (page-in rows from the host store, then the rest of each
    // paged row) or the HBM items (resident members' rows).
    auto run_items = [&](const bool as_link, int first_cta, int nctas) {
        const long long total = as_link ? link_items : hbm_items;
        {
            for (long long item = (long long)first_cta * kWp + warp; item < total; item += (long long)nctas * kWp) {
                if (as_link && item >= miss_rows) {
                    const long long c = item - miss_rows;
                    const int m = (int)(c / copies_per);
                    const size_t off = s.tail_off + (size_t)(c - (long long)m * copies_per) * kCopyItem;
                    const uint8_t* src = host + (size_t)sh_mexp[m] * s.stride + off;
                    uint8_t* dst = slots + (size_t)sh_mslot[m] * s.stride + off;
                    const size_t nbytes = min(kCopyItem, s.copy_bytes - off);
                    int4 v[kCopyLd];
#pragma unroll
                    for (int u = 0; u < kCopyLd; ++u) {
                        const size_t o = ((size_t)u * 32 + lane) * 16;
                        if (o < nbytes) v[u] = ld_nc_na(src + o);
                    }
#pragma unroll
                    for (int u = 0; u < kCopyLd; ++u) {
                        const size_t o = ((size_t)u * 32 + lane) * 16;
                        if (o < nbytes) *reinterpret_cast<int4*>(dst + o) = v[u];
                    }
                    continue;
                }
                const int mq = as_link ? (int)(item / s.I) : count + (int)(item / ipe);
                const int n = as_link ? (int)(item % s.I) : (int)(item % ipe) * RPI;  // first row pair of the item
                const int nr = as_link ? 1 : RPI;                                       // row pairs of the item
                const int slot = sh_mslot[mq];
                if constexpr (FMT == PE_MXFP4 || FMT == PE_NVFP4) {
                    uint8_t* slot_base = slots + (size_t)slot * s.stride;
                    const uint8_t* rbase = as_link ? host + (size_t)sh_mexp[mq] * s.stride : slot_base;
                    const int nch4 = s.H >> 5;
                    int4 gv[RPI][CPLH4], uv[RPI][CPLH4];
                    float2 sg[RPI][CPLH4], su[RPI][CPLH4];
#pragma unroll
                    for (int r = 0; r < RPI; ++r)
                        if (r < nr)
                            load_row_pair_fp4<FMT, CPLH4>(rbase, s, n + r, lane, nch4, as_link, false, gv[r], uv[r],
                                                          sg[r], su[r]);
                    if (as_link) {
                        uint8_t* gd = slot_base + s.w13_off + (size_t)n * (s.H / 2);
                        uint8_t* ud = gd + (size_t)s.I * (s.H / 2);
#pragma unroll
                        for (int c = 0; c < CPLH4; ++c) {
                            const int idx = lane + 32 * c;
                            if (idx < nch4) {
                                *reinterpret_cast<int4*>(gd + 16 * (size_t)idx) = gv[0][c];
                                *reinterpret_cast<int4*>(ud + 16 * (size_t)idx) = uv[0][c];
                            }
                        }
                    }
                    for (int b0 = 0; b0 < nent; b0 += 32) {
                        const int i = b0 + lane;
                        unsigned mask = __ballot_sync(0xffffffffu, i < nent && sh_ekey[i] == slot);
                        while (mask) {
                            const int ei = b0 + __ffs(mask) - 1;
                            mask &= mask - 1;
                            const uint8_t* xr = xbase + (size_t)(ei / s.k) * s.H * 2;
#pragma unroll
                            for (int r = 0; r < RPI; ++r) {
                                if (r >= nr) break;
                                const float hval = row_pair_h_fp4<CPLH4>(gv[r], uv[r], sg[r], su[r], xr, lane, nch4);
                                if (lane == 0) hbuf[(size_t)ei * s.I + n + r] = hval;
                            }
                        }
                    }
                    continue;
                }
                if constexpr (FMT == PE_INT4_GPTQ) {
                    uint8_t* slot_base = slots + (size_t)slot * s.stride;
                    const uint8_t* rbase = as_link ? host + (size_t)sh_mexp[mq] * s.stride : slot_base;
                    const int nch4 = s.H >> 5;
                    int4 gv[RPI][CPLH4], uv[RPI][CPLH4];
                    float sg[RPI][CPLH4], su[RPI][CPLH4];
#pragma unroll
                    for (int r = 0; r < RPI; ++r)
                        if (r < nr)
                            load_row_pair_int4<CPLH4>(rbase, s, n + r, lane, nch4, as_link, false, gv[r], uv[r], sg[r],
                                                      su[r]);
                    if (as_link) {
#pragma unroll
                        for (int r = 0; r < 1; ++r) {
                            uint8_t* gd = slot_base + s.w13_off + (size_t)(n + r) * (s.H / 2);
                            uint8_t* ud = gd + (size_t)s.I * (s.H / 2);
#pragma unroll
                            for (int c = 0; c < CPLH4; ++c) {
                                const int idx = lane + 32 * c;
                                if (idx < nch4) {
                                    *reinterpret_cast<int4*>(gd + 16 * (size_t)idx) = gv[r][c];
                                    *reinterpret_cast<int4*>(ud + 16 * (size_t)idx) = uv[r][c];
                                }
                            }
                        }
                    }
                    for (int b0 = 0; b0 < nent; b0 += 32) {
                        const int i = b0 + lane;
                        unsigned mask = __ballot_sync(0xffffffffu, i < nent && sh_ekey[i] == slot);
                        while (mask) {
                            const int ei = b0 + __ffs(mask) - 1;
                            mask &= mask - 1;
                            const uint8_t* xr = xbase + (size_t)(ei / s.k) * s.H * 2;
#pragma unroll
                            for (int r = 0; r < RPI; ++r) {
                                if (r >= nr) break;
                                const float hval = row_pair_h_int4<CPLH4>(gv[r], uv[r], sg[r], su[r], xr, lane, nch4);
                                if (lane == 0) hbuf[(size_t)ei * s.I + n + r] = hval;
                            }
                        }
                    }
                    continue;
                }
                if constexpr (FMT == PE_FP8_BLOCK128) {
                    uint8_t* slot_base = slots + (size_t)slot * s.stride;
                    const uint8_t* rbase = as_link ? host + (size_t)sh_mexp[mq] * s.stride : slot_base;
                    const int nch8 = s.H >> 4;
                    int4 gv[CPLH8], uv[CPLH8];
                    float sg[CPLH8], su[CPLH8];
                    load_row_pair_fp8<CPLH8>(rbase, s, n, lane, nch8, as_link, gv, uv, sg, su);
                    if (as_link) {
                        uint8_t* gd = slot_base + s.w13_off + (size_t)n * s.H;
                        uint8_t* ud = gd + (size_t)s.I * s.H;
#pragma unroll
                        for (int c = 0; c < CPLH8; ++c) {
                            const int idx = lane + 32 * c;
                            if (idx < nch8) {
                                *reinterpret_cast<int4*>(gd + 16 * (size_t)idx) = gv[c];
                                *reinterpret_cast<int4*>(ud + 16 * (size_t)idx) = uv[c];
                            }
                        }
                    }
                    for (int b0 = 0; b0 < nent; b0 += 32) {
                        const int i = b0 + lane;
                        unsigned mask = __ballot_sync(0xffffffffu, i < nent && sh_ekey[i] == slot);
                        while (mask) {
                            const int ei = b0 + __ffs(mask) - 1;
                            mask &= mask - 1;
                            const float hval = row_pair_h_fp8<CPLH8>(gv, uv, sg, su,
                                                                     xbase + (size_t)(ei / s.k) * s.H * 2, lane, nch8);
                            if (lane == 0) hbuf[(size_t)ei * s.I + n] = hval;
                        }
                    }
                    continue;
                }
                uint8_t* slot_row = slots + (size_t)slot * s.stride + s.w13_off;
                const uint8_t* g = (as_link ? host + (size_t)sh_mexp[mq] * s.stride + s.w13_off : slot_row) +
                                   (size_t)n * row_bytes;
                const uint8_t* u = g + (size_t)s.I * row_bytes;
                int4 gv[CPLH], uv[CPLH];
#pragma unroll
                for (int c = 0; c < CPLH; ++c) {
                    const int idx = lane + 32 * c;
                    if (idx < nchunk) {
                        gv[c] = as_link ? ld_nc_na(g + 16 * (size_t)idx) : ldg16(g + 16 * (size_t)idx);
                        uv[c] = as_link ? ld_nc_na(u + 16 * (size_t)idx) : ldg16(u + 16 * (size_t)idx);
                    } else {
                        gv[c] = uv[c] = make_int4(0, 0, 0, 0);
                    }
                }
                if (as_link) {
                    uint8_t* gd = slot_row + (size_t)n * row_bytes;
                    uint8_t* ud = gd + (size_t)s.I * row_bytes;
#pragma unroll
                    for (int c = 0; c < CPLH; ++c) {
                        const int idx = lane + 32 * c;
                        if (idx < nchunk) {
                            *reinterpret_cast<int4*>(gd + 16 * (size_t)idx) = gv[c];
                            *reinterpret_cast<int4*>(ud + 16 * (size_t)idx) = uv[c];
                        }
                    }
                }
                for (int b0 = 0; b0 < nent; b0 += 32) {
                    const int i = b0 + lane;
                    unsigned mask = __ballot_sync(0xffffffffu, i < nent && sh_ekey[i] == slot);
                    while (mask) {
                        const int ei = b0 + __ffs(mask) - 1;
                        mask &= mask - 1;
                        const float hval =
                            row_pair_h<CPLH>(gv, uv, xbase + (size_t)(ei / s.k) * row_bytes, lane, nchunk);
                        if (lane == 0) hbuf[(size_t)ei * s.I + n] = hval;
                    }
                }
            }
        }
    };

    // ---- phase 1 ----
    if (link_cta) {
        run_items(true, rank, link_ctas);
        cta_arrive(&sync[D_LINK]);
    }
    if (hbm_cta) {
        run_items(false, rank, hbm_ctas);
        cta_arrive(&sync[D_HITS]);
    }

    // Down items read the entry's h from shared memory: the eight warps of a
    // CTA take eight consecutive down items of one entry, and the CTA stages
    // that entry's h once for all of them (hs_pos layout, F4 float4s per
    // lane chunk) rather than every warp reading it through L2.
    constexpr int F4 = is_4bit(FMT) ? 8 : FMT == PE_FP8_BLOCK128 ? 4 : 2;
    float* sh_h = reinterpret_cast<float*>(sh_mexp + decode_meta_words(s));
    auto stage_h = [&](int e) {
        const float4* src = reinterpret_cast<const float4*>(hbuf + (size_t)e * s.I);
        float4* dst = reinterpret_cast<float4*>(sh_h);
        for (int i = threadIdx.x; i < s.I / 4; i += kThr) dst[hs_pos<F4>(i / F4, i % F4)] = __ldcg(src + i);
    };
    // down projection rows m0.. of entry e into the merged buffer
    auto down_entry = [&](int e, int m0) {
        const uint8_t* sb = slots + (size_t)sh_ekey[e] * s.stride;
        const float we = sh_ew[e];
        if constexpr (FMT == PE_MXFP4 || FMT == PE_NVFP4)
            down_rows_fp4<FMT, CPLI4, RD, true, true>(sb + s.w2_off, sb + s.s2_off, sh_h, we, m0, s.H, s.I, true,
                                                merged + (size_t)e * s.H, nullptr, lane);
        else if constexpr (FMT == PE_INT4_GPTQ)
            down_rows_int4<CPLI4, RD, true, true>(sb + s.w2_off, reinterpret_cast<const __half*>(sb + s.s2_off), sh_h, we,
                                            m0, s.H, s.I, true, merged + (size_t)e * s.H, nullptr, lane);
        else if constexpr (FMT == PE_FP8_BLOCK128)
            down_rows_fp8<CPLI8>(sb + s.w2_off, reinterpret_cast<const float*>(sb + s.s2_off), sh_h, we, m0, s.H,
                                 s.I, merged + (size_t)e * s.H, lane);
        else
            down_rows<CPLI>(sb + s.w2_off, sh_h, we, m0, s.H, s.I, merged + (size_t)e * s.H, lane);
    };

    // ---- phase 2: down projections ----
    // Down items are numbered per entry in blocks of kWp (row blocks padded to
    // a multiple of kWp), so the kWp items a CTA takes at once, one per warp,
    // belong to one entry.
    const long long rbp = (row_blocks + kWp - 1) / kWp * kWp;
    // Resident experts: as soon as every resident expert's h is done.  Items
    // go out eight at a time (one per warp) from a per-step ticket, so link
    // CTAs that finish their page-ins early (small or few page-ins) help.
    if (hbm_cta || hbm_items > 0) {
        cta_wait(&sync[D_HITS], (unsigned)hbm_ctas, err, &sh_flag);
        const long long items = (long long)sh_nhit * rbp;
        __shared__ unsigned sh_ticket;
        for (;;) {
            // every warp is done with the previous items (and their staged h)
            if (threadIdx.x == 0) sh_ticket = atomicAdd(&sync[H_TICKET], (unsigned)kWp);
            __syncthreads();
            const long long base = sh_ticket;
            if (base < items) stage_h(sh_hit_list[base / rbp]);
            __syncthreads();  // h staged, and every warp has read the ticket before thread 0 takes the next
            if (base >= items) break;
            const long long it = base + warp;
            const int blk = (int)(it % rbp);
            if (blk < row_blocks) down_entry(sh_hit_list[it / rbp], blk * RD);
        }
    }
    // paged experts: once the link is drained (their h and their w2 rows)
    cta_wait(&sync[D_LINK], (unsigned)link_ctas, err, &sh_flag);
    {
        const long long items = (long long)sh_nmiss * rbp;
        for (long long base = (long long)blockIdx.x * kWp; base < items; base += (long long)G * kWp) {
            __syncthreads();  // every warp is done with the previous items' staged h
            stage_h(sh_miss_list[base / rbp]);
            __syncthreads();
            const long long it = base + warp;
            const int blk = (int)(it % rbp);
            if (blk < row_blocks) down_entry(sh_miss_list[it / rbp], blk * RD);
        }
    }
    cta_arrive(&sync[S_DOWN]);
    cta_wait(&sync[S_DOWN], (unsigned)G, err, &sh_flag);
    pdl_trigger();

    // ---- phase 3: top-k sum in entry order ----
    const long long total = (long long)T * s.H;
    for (long long q = (long long)blockIdx.x * blockDim.x + threadIdx.x; q < total; q += (long long)G * blockDim.x) {
        const int t = (int)(q / s.H);
        const int m = (int)(q - (long long)t * s.H);
        float acc = 0.f;
        for (int j = 0; j < s.k; ++j) acc = __fadd_rn(acc, __ldcg(merged + ((size_t)t * s.k + j) * s.H + m));
        out[q] = __float2bfloat16_rn(acc);
    }

    // the last CTA out resets the counters for this layer's next step
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(&sync[S_EXIT], 1u) == (unsigned)G - 1) {
            for (int i = 0; i < S_EXIT; ++i) sync[i] = 0;
            __threadfence();
            sync[S_EXIT] = 0;
        }
    }
}

// Self-test: a phase wait on a counter nothing increments must give up.
__global__ void decode_wait_selftest_kernel(const unsigned* never, uint32_t* err, uint32_t limit) {
    __shared__ int sh_flag;
    cta_wait(never, 1u, err, &sh_flag, limit);
}

}  // namespace

cudaError_t selftest_decode_wait(const unsigned* never, uint32_t* err, uint32_t limit, cudaStream_t st) {
    decode_wait_selftest_kernel<<<1, 128, 0, st>>>(never, err, limit);
    return cudaGetLastError();
}

int decode_fused_sync_words() { return S_NUM; }

bool decode_fused_supported(const Shape& s, int T) {
    const bool dims = s.dtype == PE_FP8_BLOCK128 ? (s.H <= 32 * 16 * CPLH8 && s.I <= 32 * 16 * CPLI8)
                      : is_4bit(s.dtype) ? (s.H <= 32 * 32 * CPLH4 && s.I <= 32 * 32 * CPLI4)
                                                : (s.H <= 32 * 8 * CPLH && s.I <= 32 * 8 * CPLI);
    return (long long)T * s.k <= kFusedMaxEntries && (long long)T * s.k <= s.K && s.E <= kPlanCap &&
           s.K <= kPlanCap && dims &&
           (size_t)4 * (decode_meta_words(s) + decode_hstage_words(s)) <= (size_t)kDynBudget;
}

cudaError_t decode_setup_kernels() {
    cudaError_t e = cudaSuccess;
#define PE_ATTR(N)                                                                                                   \
    if (!e) e = cudaFuncSetAttribute(decode_step_kernel<N, PE_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynBudget); \
    if (!e) e = cudaFuncSetAttribute(decode_step_kernel<N, PE_FP8_BLOCK128>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynBudget); \
    if (!e) e = cudaFuncSetAttribute(decode_step_kernel<N, PE_INT4_GPTQ>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynBudget); \
    if (!e) e = cudaFuncSetAttribute(decode_step_kernel<N, PE_MXFP4>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynBudget); \
    if (!e) e = cudaFuncSetAttribute(decode_step_kernel<N, PE_NVFP4>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynBudget);
    PE_ATTR(1) PE_ATTR(2) PE_ATTR(4) PE_ATTR(8)
#undef PE_ATTR
    return e;
}

cudaError_t decode_ctas_per_sm(int dtype, int* out) {
    // The phase counters need every CTA of the grid resident at once, so the
    // grid is (resident CTAs per SM, at most 2) x SMs, taken at the largest
    // dynamic shared memory a launch may ask for and over every instantiation
    // of the format.
    int best = 2;
    cudaError_t e = cudaSuccess;
#define PE_OCC(N, F)                                                                                              \
    if (!e) {                                                                                                     \
        int n = 0;                                                                                                \
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_step_kernel<N, F>, kThr, kDynBudget);        \
        if (!e && n < best) best = n;                                                                             \
    }
#define PE_OCC_F(F) PE_OCC(1, F) PE_OCC(2, F) PE_OCC(4, F) PE_OCC(8, F)
    if (dtype == PE_FP8_BLOCK128) {
        PE_OCC_F(PE_FP8_BLOCK128)
    } else if (dtype == PE_INT4_GPTQ) {
        PE_OCC_F(PE_INT4_GPTQ)
    } else if (dtype == PE_MXFP4) {
        PE_OCC_F(PE_MXFP4)
    } else if (dtype == PE_NVFP4) {
        PE_OCC_F(PE_NVFP4)
    } else {
        PE_OCC_F(PE_BF16)
    }
#undef PE_OCC_F
#undef PE_OCC
    *out = e ? 0 : best;
    return e;
}

cudaError_t launch_decode_fused(const LayerDev& L, const Shape& s, const float* logits, const __nv_bfloat16* x,
                                const uint8_t* host_layer, uint8_t* slots_layer, int T, float* hbuf, float* merged,
                                __nv_bfloat16* out, unsigned* sync, uint32_t* err, int num_sms, int ctas_per_sm,
                                cudaStream_t st) {
    const int grid = num_sms * ctas_per_sm;  // every CTA is resident at once (decode_ctas_per_sm)
    const size_t meta = (size_t)4 * (decode_meta_words(s) + decode_hstage_words(s));
    const size_t xbytes = (size_t)T * s.H * 2;
    const int stage = meta + xbytes <= (size_t)kDynBudget;
    const size_t smem = meta + (stage ? xbytes : 0);
    const int epl = (s.E + 31) / 32;
#define PE_DEC1(N, F)                                                                                               \
    launch_pdl(decode_step_kernel<N, F>, grid, kThr, smem, st, L, s, logits, x, host_layer, slots_layer, T, hbuf,     \
               merged, out, sync, err, stage)
#define PE_DEC(N)                                                                                                   \
    return s.dtype == PE_FP8_BLOCK128 ? PE_DEC1(N, PE_FP8_BLOCK128)                                                 \
           : s.dtype == PE_INT4_GPTQ  ? PE_DEC1(N, PE_INT4_GPTQ)                                                    \
           : s.dtype == PE_MXFP4      ? PE_DEC1(N, PE_MXFP4)                                                        \
           : s.dtype == PE_NVFP4      ? PE_DEC1(N, PE_NVFP4)                                                        \
                                      : PE_DEC1(N, PE_BF16)
    if (epl <= 1) PE_DEC(1);
    if (epl <= 2) PE_DEC(2);
    if (epl <= 4) PE_DEC(4);
    PE_DEC(8);
#undef PE_DEC
#undef PE_DEC1
}

}  // namespace pe
