// Internal declarations shared by the libpe translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pe.h"

namespace pe {

constexpr int kMaxExperts = 1024;  // plan kernel keeps per-expert flags in shared memory
constexpr int kMaxSlots = 1024;
constexpr int kMaxTopK = 32;       // one warp lane per chosen expert
constexpr int kPlanMaxThreads = 1024;
constexpr int kFusedMaxEntries = 64;  // decode: one warp scans a wave's entries per weight row
constexpr int kFp8Block = 128;
constexpr int kInt4Group = 128;  // GPTQ int4: inputs per scale
constexpr int kMxfp4Block = 32;  // MXFP4: inputs per E8M0 scale
constexpr int kNvfp4Block = 16;  // NVFP4: inputs per E4M3 scale
// The 4-bit formats (GPTQ int4, MXFP4, NVFP4) share one code layout: two
// codes per byte, rows of K/2 bytes.
__host__ __device__ constexpr bool is_4bit(int dtype) {
    return dtype == PE_INT4_GPTQ || dtype == PE_MXFP4 || dtype == PE_NVFP4;
}
// Shape of one prefill GEMM tile.  Token rows sit on the MMA's M (TMEM
// lanes), weight rows on its N: a gate/up tile reads BN/2 gate and BN/2 up
// rows of w13, a down tile BN rows of w2 (the weight tensor maps' box
// heights).  bf16 tiles are 128 token rows x 256 weight rows, one M=128,
// N=256 MMA per 16-deep slice; the quantised formats, whose code staging
// takes shared memory, 256 token rows x 128 weight rows, two M=128, N=128
// MMAs sharing the weight tile.
__host__ __device__ constexpr int prefill_bn(int dtype) { return dtype == PE_BF16 ? 256 : 128; }
__host__ __device__ constexpr int prefill_mt(int dtype) { return dtype == PE_BF16 ? 128 : 256; }

enum Counter { C_STEPS = 0, C_WAVES, C_ENTRIES, C_DISTINCT, C_HITS, C_PAGE_INS, C_COLD, C_NUM };

// Device pointers of one layer's residency state and last plan.
struct LayerDev {
    int32_t* slot_expert;   // [K]   expert held by each slot, -1 = empty
    uint32_t* slot_tick;    // [K]   clock value of the slot's last use
    int32_t* expert_slot;   // [E]   slot holding each expert, -1 = not resident
    uint32_t* clock;        // [1]
    unsigned long long* counters;  // [C_NUM]
    int32_t* plan_expert;   // [Wmax][K]
    int32_t* plan_slot;     // [Wmax][K]
    int32_t* plan_count;    // [Wmax]
    int32_t* member_expert; // [Wmax][K] wave members: the page-ins (plan order), then the hits
    int32_t* member_slot;   // [Wmax][K] slot of each member while its wave runs
    int32_t* member_count;  // [Wmax]
    int32_t* num_waves;     // [1]
    int32_t* topk_id;       // [maxT*k]
    float* topk_w;          // [maxT*k]
    int32_t* entry_slot;    // [maxT*k]
    int32_t* entry_wave;    // [maxT*k]
    const uint8_t* loaded;  // [E]   1 once the expert's host row was written
    unsigned* dsync;        // [16]  queues and phase counters of the one-kernel decode step (zero between steps)
};

struct Shape {
    int E, k, K, H, I, Wmax;
    int dtype;
    size_t stride;       // bytes between expert rows (slot or host store)
    size_t copy_bytes;   // bytes a page-in moves (payload rounded up to 16)
    size_t w13_off, s13_off, w2_off, s2_off;
    size_t tail_off;     // start of everything after w13 (scales, w2): copied as one block
};

// Workspace of the tensor-core prefill path (rows grouped by expert, each
// expert padded to a multiple of 128 rows).
struct PrefillDev {
    __nv_bfloat16* x_perm;  // [max_rows][H]  A operand of the gate/up GEMM
    __nv_bfloat16* h_perm;  // [max_rows][I]  A operand of the down GEMM
    int32_t* perm;          // [max_rows]     entry of each row, -1 = padding
    int4* tiles;            // [max_tiles]    (row0, slot in the whole table, valid rows, member)
    int2* items;            // [max_items]    GEMM queue: (tile, kind << 16 | column tile), kind 1 = down
    int4* members;          // [E]            (expert, slot, wave, 1 if paged in) in queue order
    int32_t* pin_member;    // [E]            page-ins in plan order -> member
    int32_t* slot_need;     // [E]            GEMM tiles of the slot's earlier occupants before the page-in
    unsigned* landed;       // [E]            landed page-in chunks per member
    unsigned* gu_done;      // [max_tiles]    finished gate/up tiles per row tile
    unsigned* slot_done;    // [K]            finished GEMM tiles per slot in this step
    unsigned* ctl;          // [4]            GEMM ticket, abort word, link / GEMM CTAs registered
    int32_t* counts;        // [8]            tiles, rows, items, members, page-ins, staged members to commit
    int32_t* stage_of;      // [E]            staging row of a member paged in through staging, else -1
    int32_t* commit_member; // [E]            staged members that are their slot's last occupant in the step
    int max_rows, max_tiles, max_items;
    int stage_base;         // whole-table slot index of staging row 0 (the rows follow the L*K slots)
    int stage_rows;         // staging rows (0: no staging)
};

// TMA descriptors of the prefill path, encoded once at creation.
struct PrefillMaps {
    CUtensorMap x_perm;  // 2-D bf16 [max_rows][H], 64 x 128 boxes
    CUtensorMap h_perm;  // 2-D bf16 [max_rows][I], 64 x 128 boxes
    CUtensorMap w13;     // 3-D [L*K slots][2I][H], boxes of BN/2 rows: bf16 64 x 128 x 1 (swizzled),
                         //   FP8 codes 64 x 64 x 1, 4-bit codes [..][2I][H/2 bytes] 32 x 64 x 1
    CUtensorMap w2;      // 3-D [L*K slots][H][I], boxes of BN rows: bf16 64 x 256 x 1 (swizzled),
                         //   FP8 codes 64 x 128 x 1, 4-bit codes [..][H][I/2 bytes] 32 x 128 x 1
};

bool prefill_tc_supported(const Shape& s);
size_t prefill_max_rows(int max_entries, int E);
size_t prefill_max_tiles(int max_entries, int E);
size_t prefill_max_items(const Shape& s, size_t max_tiles);
cudaError_t prefill_setup_kernels();
// CTAs of the prefill step kernel for this format that fit on one SM (its
// grid is one CTA per SM, all resident at once; call after
// prefill_setup_kernels).
cudaError_t prefill_step_ctas_per_sm(int dtype, int* out);
// Prefill step, part 1 (after the planner): lay out every wave's members,
// tiles, GEMM queue and page-in list, and gather the token rows (align +
// gather kernels).
cudaError_t launch_prefill_align(const LayerDev& L, const Shape& s, const PrefillDev& P, const __nv_bfloat16* x,
                                 int slot_base, int T, int num_sms, cudaStream_t st);
// Prefill step, part 2: every wave's page-in and tensor-core GEMMs in one
// persistent kernel (merged entries; the top-k sum runs after it).
cudaError_t launch_prefill_step(const LayerDev& L, const Shape& s, const PrefillDev& P, const PrefillMaps& M,
                                const uint8_t* host_layer, uint8_t* slots_all, int slot_base, float* merged,
                                uint32_t* err, int num_sms, cudaStream_t st);

// Self-tests of the bounded waits (each wait runs on a condition that never
// becomes true and must give up after `limit` polls, recording the timeout).
cudaError_t selftest_decode_wait(const unsigned* never, uint32_t* err, uint32_t limit, cudaStream_t st);
cudaError_t selftest_prefill_waits(const unsigned* never, unsigned* abort_w, uint32_t* err_counter,
                                   uint32_t* err_mbar, uint32_t limit, cudaStream_t st);

// Records the message pe_last_error(NULL) returns in this thread.
void set_thread_error(const char* msg);

// ---- launchers (each returns the launch status) ----

// Routing of T tokens by one warp per token into topk_id / topk_w.
cudaError_t launch_route(const LayerDev& L, const Shape& s, const float* logits, int T,
                         uint32_t* err, cudaStream_t st);
// LRU planning of all waves of one step (one CTA); routes inline when
// route_inline is set (small T), else reads topk_id / topk_w.
cudaError_t launch_plan(const LayerDev& L, const Shape& s, const float* logits, int T,
                        int route_inline, uint32_t* err, cudaStream_t st);
// Copy the experts planned for wave `wave` from the host store into slots.
cudaError_t launch_pagein(const LayerDev& L, const Shape& s, const uint8_t* host_layer,
                          uint8_t* slots_layer, int wave, int max_count, int num_sms,
                          cudaStream_t st);
// Plain device-side copy used by the host-link probe.
cudaError_t launch_copy(const void* src, void* dst, size_t bytes, int num_sms, cudaStream_t st);
// Decode expert MLP, part 1 fused with page-in: for every member of the wave,
// stream its gate/up rows (from the host store for page-ins, which are also
// written to their slot; from the slot for hits) and compute h for every
// entry routed to it; the rest of each paged row is copied alongside.
cudaError_t launch_gateup_pagein(const LayerDev& L, const Shape& s, const __nv_bfloat16* x,
                                 const uint8_t* host_layer, uint8_t* slots_layer, int wave, int T,
                                 float* hbuf, int num_sms, cudaStream_t st);
// Decode expert MLP, part 1: h = SiLU(gate x) * (up x) for the wave's entries.
cudaError_t launch_gateup(const LayerDev& L, const Shape& s, const __nv_bfloat16* x,
                          const uint8_t* slots_layer, int wave, int T, float* hbuf,
                          int num_sms, cudaStream_t st);
// Decode expert MLP, part 2: w * (down h).  fused: sum the top-k in place
// and write out (single wave); else write merged[entry] for the wave.
cudaError_t launch_down(const LayerDev& L, const Shape& s, const uint8_t* slots_layer, int wave,
                        int T, const float* hbuf, float* merged, __nv_bfloat16* out, int fused,
                        int num_sms, cudaStream_t st);
// Single-wave decode (tokens * top_k <= min(K, kFusedMaxEntries), bf16,
// E and K <= 256): routing, plan, page-in, gate/up, down and top-k sum in one
// kernel.
bool decode_fused_supported(const Shape& s, int T);
int decode_fused_sync_words();
cudaError_t decode_setup_kernels();
// Resident CTAs per SM of the decode step kernel for this format, capped at
// 2 (its grid is this many CTAs per SM, all resident at once; call after
// decode_setup_kernels).  0 means it cannot run.
cudaError_t decode_ctas_per_sm(int dtype, int* out);
cudaError_t launch_decode_fused(const LayerDev& L, const Shape& s, const float* logits, const __nv_bfloat16* x,
                                const uint8_t* host_layer, uint8_t* slots_layer, int T, float* hbuf, float* merged,
                                __nv_bfloat16* out, unsigned* sync, uint32_t* err, int num_sms, int ctas_per_sm,
                                cudaStream_t st);

// Block-FP8 counterparts of the three decode kernels above.
cudaError_t launch_gateup_pagein_fp8(const LayerDev& L, const Shape& s, const __nv_bfloat16* x,
                                     const uint8_t* host_layer, uint8_t* slots_layer, int wave, int T,
                                     float* hbuf, int num_sms, cudaStream_t st);
cudaError_t launch_gateup_fp8(const LayerDev& L, const Shape& s, const __nv_bfloat16* x,
                              const uint8_t* slots_layer, int wave, int T, float* hbuf, int num_sms,
                              cudaStream_t st);
cudaError_t launch_down_fp8(const LayerDev& L, const Shape& s, const uint8_t* slots_layer, int wave,
                            int T, const float* hbuf, float* merged, __nv_bfloat16* out, int fused,
                            int num_sms, cudaStream_t st);
// 4-bit (GPTQ int4, MXFP4, NVFP4; chosen by s.dtype) counterparts of the
// three decode kernels above.
cudaError_t launch_gateup_pagein_q4(const LayerDev& L, const Shape& s, const __nv_bfloat16* x,
                                    const uint8_t* host_layer, uint8_t* slots_layer, int wave, int T,
                                    float* hbuf, int num_sms, cudaStream_t st);
cudaError_t launch_gateup_q4(const LayerDev& L, const Shape& s, const __nv_bfloat16* x,
                             const uint8_t* slots_layer, int wave, int T, float* hbuf, int num_sms,
                             cudaStream_t st);
cudaError_t launch_down_q4(const LayerDev& L, const Shape& s, const uint8_t* slots_layer, int wave,
                           int T, const float* hbuf, float* merged, __nv_bfloat16* out, int fused,
                           int num_sms, cudaStream_t st);
// out[t] = sum_j merged[t, j] in entry order, rounded to bf16.
cudaError_t launch_topk_sum(const Shape& s, const float* merged, __nv_bfloat16* out, int T,
                            cudaStream_t st);

}  // namespace pe
