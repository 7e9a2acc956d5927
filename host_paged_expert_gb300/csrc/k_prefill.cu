// Prefill-sized layer step: page-in and the expert MLP on the tcgen05 tensor
// cores, pipelined in one persistent kernel.
//
// "Paged Experts" (SGLang docs), "A step: waves, page-in, merge": a step
// whose distinct experts exceed the slots runs in waves; each wave pages in
// its missing experts, runs the fused-MoE kernel over the wave's own entries
// (each output multiplied by its router weight, no top-k sum), and the merged
// entries are summed once after the last wave.  At prefill sizes an expert has
// tens to hundreds of routed tokens, so its MLP is a pair of dense
// contractions:
//   GEMM1: [rows_e, H] x w13[2I, H]^T  -> SiLU(gate) * up -> h [rows_e, I] (bf16)
//   GEMM2: [rows_e, I] x w2[H, I]^T    -> * router weight -> merged entries (fp32)
//
// After the planner, a layer step is three kernels:
//   align   (one CTA) lays out every member of every wave: a packed row range
//           per member (padded to 128 rows), the row -> entry map, a tile
//           table, the GEMM work queue, the page-in list, the staging rows
//           (below), and for each member how many GEMM tiles of its slot's
//           earlier occupants in this step must finish before the slot may
//           be overwritten;
//   gather  copies each entry's token row of x into the packed A operand;
//   step    one persistent CTA per SM.  The CTA on every fourth SM streams
//           the host link: it copies 64 KiB chunks of the planned experts, in plan
//           order, from the pinned host store into their slots and counts
//           each expert's landed chunks, then joins the GEMM CTAs.  Those
//           take GEMM tiles from a queue in the same order (the hits of
//           wave 0 first, each expert's down tiles trailing its gate/up
//           tiles by two rounds of the GEMM CTAs within its wave): a
//           gate/up tile starts once every chunk of its expert has landed, a
//           down tile once all gate/up tiles of its rows are done.  So the
//           resident experts compute while the misses page in, every paged
//           expert computes as soon as it has landed, and wave w+1's page-in
//           runs under wave w's GEMMs.
// A page-in whose slot an earlier wave's expert still uses streams into one
// of K staging rows after the slot table instead of waiting (the first K
// such, in plan order; the others wait for the slot): its tiles read the
// staging row, and if it is the slot's last occupant in the step, a link CTA
// copies the row into the slot once every tile that reads the slot is done.
// The waves, the residency after the step and the results stay exactly the
// planner's: nothing overwrites a slot before the GEMMs that read it are done.
//
// A GEMM tile is up to 256 rows of one expert x 128 output columns.  A GEMM
// CTA is a pipeline of warp roles that hand tiles on through mbarriers:
//   warp 0      scheduler and TMA producer: takes the next tile, waits for
//               what it reads, publishes it to the other roles (a 4-deep
//               queue) and streams its k-steps (128-byte-swizzled A and B
//               tiles) into a 4-stage shared-memory ring;
//   warp 1      MMA issuer: two M=128 tcgen05.mma per k-step that share the
//               weight tile (the second only when the expert has more than
//               128 rows), into one of two TMEM accumulator buffers;
//   warps 2-11  converters for quantised weights (below);
//   warps 12-15 epilogue: TMEM -> SiLU(gate)*up into h (bf16), or router
//               weight x result into the merged entries, then count the
//               tile done.
// With two accumulator buffers the MMAs of one tile run while the epilogue
// of the previous one drains, and the producer streams ahead across tiles.
// The weights come straight from the slot table (a 3-D tensor map over
// [slot][row][k]).
//
// Block-FP8 experts (E4M3 codes, one fp32 scale per 128x128 block), GPTQ
// int4 experts (4-bit codes, zero point 8, one fp16 scale per output row and
// 128 inputs) and MXFP4 / NVFP4 experts (E2M1 codes with E8M0 scales per 32
// inputs, or E4M3 scales per 16 inputs and an fp32 tensor scale) keep bf16
// activations: TMA brings the code tile into a staging buffer, ten converter
// warps decode it, multiply by its scale, round to bf16 and write it in the
// 128-byte-swizzled layout the MMA reads; the MMA then runs as for bf16.  A
// tile's scales are staged in shared memory once per tile (FP8: one row of
// blocks for each of its gate, up or down row ranges; the 4-bit formats:
// every row's scales).
//
// Every row of an MMA tile is computed independently and always with the same
// k order, so an entry's result does not depend on its tile-mates, its slot,
// its wave or the pipeline's timing: paged and unpaged prefill agree bit for
// bit.
//
// Every wait is bounded.  A wait that runs out records PE_DEVERR_TIMEOUT and
// raises the step's abort word, after which every wait gives up at once; the
// work behind a failed wait is skipped but still counted as done, so the
// kernel always ends.

#include <cuda_fp16.h>

#include "fp4_device.cuh"
#include "fp8_device.cuh"
#include "int4_device.cuh"
#include "pe_device.cuh"
#include "pe_internal.h"
#include "tc_sm100.cuh"

namespace pe {
namespace {

constexpr int BM = 128, BK = 64, STAGES = 4;
constexpr int kQBN = 128;             // weight rows of a quantised tile (prefill_bn)
constexpr int A_BYTES = BM * BK * 2;  // one 128-row part of the token (A) tile
constexpr int kAccCols = 256;         // TMEM columns of one accumulator buffer
constexpr int kConvWarps = 10;        // warps 2..11: decode quantised weight tiles (idle for bf16)
constexpr int kEpiWarps = 4;          // warps 12..15: the epilogue (one per TMEM lane quarter)
constexpr int kStepThreads = (2 + kConvWarps + kEpiWarps) * 32;
constexpr int kInfoDepth = 4;         // tiles the scheduler may publish ahead
constexpr uint32_t kTmemCols = 2 * kAccCols;  // two accumulator buffers
constexpr int kLinkEvery = 4;         // the CTAs on SMs 0, 4, 8, ... stream the host link
constexpr int kLinkUnroll = 8;
constexpr size_t kLinkChunk = (size_t)kStepThreads * 16 * kLinkUnroll;  // 64 KiB per item
constexpr int kMaxScaleCols = 64;     // FP8 / int4: K / 128 of either GEMM (H, I <= 8192)
constexpr int kScaleStageBytes = kQBN * kMaxScaleCols * 2;  // a 4-bit tile's staged scales: 16 KiB
constexpr uint32_t kSpin = 1u << 22;  // polls, >= 128 ns apart

// Stage layout per weight format (PE_BF16, PE_FP8_BLOCK128, the 4-bit formats):
// [A part 0 (token rows 0-127)][A part 1 (rows 128-255; quantised formats)]
// [B tile, bf16, swizzled][quantised formats only: code staging], every part
// 1024-aligned.
template <int FMT>
struct Tile {
    static constexpr int BN = prefill_bn(FMT);       // weight rows (MMA N)
    static constexpr int MT = prefill_mt(FMT);       // token rows (one or two M=128 MMAs)
    static constexpr int A_PARTS = MT / BM;          // 128-row token boxes per k-step
    static constexpr int B_BYTES = BN * BK * 2;      // the bf16 weight tile
    static constexpr int C_BYTES = FMT == PE_FP8_BLOCK128 ? BN * BK          // E4M3 codes of the weight tile
                                   : is_4bit(FMT)         ? BN * BK / 2      // 4-bit codes of the weight tile
                                                          : 0;
    static constexpr int STAGE_BYTES = A_PARTS * A_BYTES + B_BYTES + C_BYTES;
    static constexpr int SMEM = STAGES * STAGE_BYTES + 1024;  // + slack to align the ring
    static_assert(A_PARTS * BN <= kAccCols, "an accumulator buffer holds the tile");
};

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Thread-level bounded wait for *p >= target.  Gives up at once when the
// step's abort word is set; running out of polls records the timeout and
// sets the abort word.
__device__ __forceinline__ int spin_geq(const unsigned* p, unsigned target, unsigned* abort_w, uint32_t* err,
                                        uint32_t limit = kSpin) {
    for (uint32_t i = 0; i < limit; ++i) {
        if (ld_acquire(p) >= target) return 1;
        if (*reinterpret_cast<volatile unsigned*>(abort_w)) return 0;
        __nanosleep(128);
    }
    atomicOr(err, PE_DEVERR_TIMEOUT);
    atomicExch(abort_w, 1u);
    return 0;
}

// ---------------------------------------------------------------- align

// Exclusive prefix sum of v over the threads of the block, in thread order;
// every thread calls it and gets the block total in *total.  sh: 32 ints.
__device__ __forceinline__ int block_excl_scan(int v, int* sh, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int t = lane < nw ? sh[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        sh[lane] = t;
    }
    __syncthreads();
    const int base = warp > 0 ? sh[warp - 1] : 0;
    *total = sh[nw - 1];
    __syncthreads();  // sh may be reused
    return base + x - v;
}

// Lays out one prefill step (one CTA of 1024 threads; E, K <= 1024, so thread
// i owns member i, slot i or page-in i in each pass).
//
// Members in queue order, wave by wave.  In each wave: first the hits whose
// slots the next wave's page-ins evict, in the order those page-ins run (so
// the link can go on to the next wave early); then the other hits; then the
// page-ins in plan order (the order they land).
//
// The GEMM queue, wave by wave: each member's gate/up tiles in member order,
// and its down tiles `lag` items later (so that a CTA taking a down tile
// rarely waits for the member's gate/up tiles), never past the end of the
// member's wave.  Every tile therefore depends only on tiles before it in
// the queue (its own member's gate/up tiles, the page-in of its expert, and
// through that page-in the tiles of earlier waves that used its slot), which
// keeps the persistent pipeline free of deadlock.
// Wave and expert of entries i0, i0 + stride, ... (kAlignBatch of them; -1
// waves past nent), all loads issued before any is used.
constexpr int kAlignBatch = 8;
__device__ __forceinline__ void load_entries(const LayerDev& L, int i0, int stride, int nent, int (&ew)[kAlignBatch],
                                             int (&id)[kAlignBatch]) {
#pragma unroll
    for (int u = 0; u < kAlignBatch; ++u) {
        const int i = i0 + u * stride;
        ew[u] = i < nent ? L.entry_wave[i] : -1;
        id[u] = i < nent ? L.topk_id[i] : 0;
    }
}

__global__ void __launch_bounds__(1024) prefill_align_kernel(LayerDev L, Shape s, PrefillDev P, int slot_base, int T,
                                                             int n1, int n2, unsigned nchunk, int lag, int MT) {
    __shared__ int sh_g_of_e[kMaxExperts];  // expert -> member
    __shared__ int sh_me[kMaxExperts], sh_ms[kMaxExperts], sh_wp[kMaxExperts];  // expert, slot, wave*2 + paged
    __shared__ int sh_cnt[kMaxExperts], sh_off[kMaxExperts], sh_fill[kMaxExperts];
    __shared__ int sh_t0[kMaxExperts + 1], sh_i0[kMaxExperts], sh_d0[kMaxExperts];  // tiles, gate/up and down queue bases
    __shared__ int sh_cum[kMaxSlots];
    __shared__ int sh_scan[32];
    // the plan's member and page-in lists, copied in parallel: [Wmax] member
    // counts, [Wmax] page-in counts, [Wmax*K] member experts, member slots,
    // page-in slots
    extern __shared__ int sh_plan[];
    int* sh_mcount = sh_plan;
    int* sh_pcount = sh_mcount + s.Wmax;
    int* sh_mexp = sh_pcount + s.Wmax;
    int* sh_mslot = sh_mexp + s.Wmax * s.K;
    int* sh_pslot = sh_mslot + s.Wmax * s.K;
    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int nent = T * s.k, K = s.K;
    const int nW = min(*L.num_waves, s.Wmax);
    for (int e = tid; e < s.E; e += nthr) sh_g_of_e[e] = -1;
    for (int i = tid; i < K; i += nthr) {
        sh_cum[i] = 0;
        P.slot_done[i] = 0;
    }
    for (int w = tid; w < nW; w += nthr) {
        sh_mcount[w] = L.member_count[w];
        sh_pcount[w] = L.plan_count[w];
    }
    for (int i = tid; i < nW * K; i += nthr) {
        sh_mexp[i] = L.member_expert[i];
        sh_mslot[i] = L.member_slot[i];
        sh_pslot[i] = L.plan_slot[i];
    }
    if (tid == 0) {
        P.ctl[0] = 0;  // GEMM ticket
        P.ctl[1] = 0;  // abort word
        P.ctl[2] = 0;  // link CTAs registered
        P.ctl[3] = 0;  // GEMM CTAs registered
    }
    __syncthreads();

    // ---- members in queue order (sh_off: slot -> member-list index of the
    // wave, sh_fill: next-wave page-in rank of a hit, sh_cnt: queue position
    // of the needed hits by that rank; all three are set afresh below)
    int gbase = 0, npbase = 0;
    for (int w = 0; w < nW; ++w) {
        const int size = sh_mcount[w], nmiss = sh_pcount[w], next = w + 1 < nW ? sh_pcount[w + 1] : 0;
        for (int i = tid; i < K; i += nthr) sh_off[i] = -1;
        if (tid < size) sh_fill[tid] = -1;
        __syncthreads();
        if (tid < size) sh_off[sh_mslot[w * K + tid]] = tid;
        __syncthreads();
        int q_of_p = -1;
        if (tid < next) {
            const int q = sh_off[sh_pslot[(w + 1) * K + tid]];
            if (q >= nmiss && q < size) {  // the next wave evicts this wave's hit q
                q_of_p = q;
                sh_fill[q] = tid;
            }
        }
        int n_needed;
        const int pos_needed = block_excl_scan(q_of_p >= 0 ? 1 : 0, sh_scan, &n_needed);
        if (q_of_p >= 0) sh_cnt[tid] = pos_needed;
        __syncthreads();
        const bool hit = tid >= nmiss && tid < size;
        const bool other = hit && sh_fill[tid] < 0;
        int n_other;
        const int pos_other = block_excl_scan(other ? 1 : 0, sh_scan, &n_other);
        if (tid < size) {
            const int q = tid, paged = q < nmiss;
            const int pos = paged ? n_needed + n_other + q : other ? n_needed + pos_other : sh_cnt[sh_fill[q]];
            const int g = gbase + pos;
            const int e = sh_mexp[w * K + q], slot = sh_mslot[w * K + q];
            sh_me[g] = e;
            sh_ms[g] = slot;
            sh_wp[g] = (w << 1) | paged;
            P.members[g] = make_int4(e, slot, w, paged);
            if (paged) {
                P.pin_member[npbase + q] = g;
                sh_i0[npbase + q] = g;  // the page-in list, until the queue bases take sh_i0 over
            }
        }
        gbase += size;
        npbase += nmiss;
        __syncthreads();
    }
    const int G = gbase;
    if (tid == 0) {
        P.counts[3] = G;
        P.counts[4] = npbase;
    }
    for (int g = tid; g < G; g += nthr) {
        sh_g_of_e[sh_me[g]] = g;
        sh_cnt[g] = 0;
        sh_fill[g] = 0;
    }
    __syncthreads();
    // entries' members, loaded kAlignBatch per thread at a time so their loads overlap
    for (int i0 = tid; i0 < nent; i0 += kAlignBatch * nthr) {
        int ew[kAlignBatch], id[kAlignBatch];
        load_entries(L, i0, nthr, nent, ew, id);
#pragma unroll
        for (int u = 0; u < kAlignBatch; ++u)
            if (ew[u] >= 0) {
                const int g = sh_g_of_e[id[u]];
                if (g >= 0) atomicAdd(&sh_cnt[g], 1);
            }
    }
    __syncthreads();

    // ---- row ranges and tiles: member g's rows are padded to 128, its tiles
    // hold up to 256 rows
    const int c = tid < G ? sh_cnt[tid] : 0;
    const int mt = (c + MT - 1) / MT;
    int rows_total, nt;
    const int off = block_excl_scan((c + BM - 1) / BM * BM, sh_scan, &rows_total);
    const int t0 = block_excl_scan(mt, sh_scan, &nt);
    if (tid < G) {
        sh_off[tid] = off;
        sh_t0[tid] = t0;
    }
    if (tid == 0) sh_t0[G] = nt;
    // Which members have an earlier occupant of their slot in this step
    // (sh_d0, for the staging choice below): members are in wave order and a
    // slot holds one member per wave.  sh_cum: slot -> occupants so far.
    {
        int wb = 0;
        for (int w = 0; w < nW; ++w) {
            const int size = sh_mcount[w];
            const bool mine = tid >= wb && tid < wb + size;
            if (mine) sh_d0[tid] = sh_cum[sh_ms[tid]];
            __syncthreads();
            if (mine) sh_cum[sh_ms[tid]] += 1;
            __syncthreads();
            wb += size;
        }
    }
    // Staging: a page-in whose slot still has an earlier occupant in this step
    // goes to a staging row (the first stage_rows such, in plan order), so the
    // link need not wait for that occupant's tiles; its tiles read the staging
    // row, and the row is copied into the slot once the slot is free if the
    // member is the slot's last occupant.  sh_d0: member -> staging row or -1.
    {
        const int np = npbase;
        int want = 0, gp = -1;
        if (tid < np) {
            gp = sh_i0[tid];
            want = sh_d0[gp] > 0;
        }
        int nwant;
        const int spos = block_excl_scan(want, sh_scan, &nwant);
        if (tid < G) sh_d0[tid] = -1;
        __syncthreads();
        if (want && spos < P.stage_rows) sh_d0[gp] = spos;
        __syncthreads();
        // GEMM tiles of each slot's earlier occupants that read the slot
        // itself (a staged member reads its staging row and is not counted),
        // then each slot's last occupant (sh_cum: slot -> member)
        for (int i = tid; i < K; i += nthr) sh_cum[i] = 0;
        __syncthreads();
        int wb = 0;
        for (int w = 0; w < nW; ++w) {
            const int size = sh_mcount[w];
            const bool mine = tid >= wb && tid < wb + size;
            if (mine) P.slot_need[tid] = sh_cum[sh_ms[tid]];
            __syncthreads();
            if (mine && sh_d0[tid] < 0) sh_cum[sh_ms[tid]] += mt * (n1 + n2);
            __syncthreads();
            wb += size;
        }
        wb = 0;
        for (int w = 0; w < nW; ++w) {
            const int size = sh_mcount[w];
            if (tid >= wb && tid < wb + size) sh_cum[sh_ms[tid]] = tid;
            __syncthreads();
            wb += size;
        }
        const bool commit = tid < G && sh_d0[tid] >= 0 && sh_cum[sh_ms[tid]] == tid;
        int ncommit;
        const int cpos = block_excl_scan(commit ? 1 : 0, sh_scan, &ncommit);
        if (commit) P.commit_member[cpos] = tid;
        if (tid == 0) P.counts[5] = ncommit;
    }
    if (tid < G) {
        const int st = sh_d0[tid];
        P.stage_of[tid] = st;
        const int slot_index = st >= 0 ? P.stage_base + st : slot_base + sh_ms[tid];
        for (int i = 0; i < mt && t0 + i < P.max_tiles; ++i)
            P.tiles[t0 + i] = make_int4(off + i * MT, slot_index, min(MT, c - i * MT), tid);
    }
    __syncthreads();  // sh_i0 and sh_d0 are the queue bases' from here on
    if (tid == 0) {
        // queue bases: gate/up blocks in member order, each down block once
        // `lag` more items have been queued, flushed at every wave's end
        int ni = 0, head = 0;
        for (int g = 0; g < G; ++g) {
            if (g > 0 && (sh_wp[g] >> 1) != (sh_wp[g - 1] >> 1))
                for (; head < g; ++head) {
                    sh_d0[head] = ni;
                    ni += (sh_t0[head + 1] - sh_t0[head]) * n2;
                }
            sh_i0[g] = ni;
            ni += (sh_t0[g + 1] - sh_t0[g]) * n1;
            for (; head < g && ni - (sh_i0[head] + (sh_t0[head + 1] - sh_t0[head]) * n1) >= lag; ++head) {
                sh_d0[head] = ni;
                ni += (sh_t0[head + 1] - sh_t0[head]) * n2;
            }
        }
        for (; head < G; ++head) {
            sh_d0[head] = ni;
            ni += (sh_t0[head + 1] - sh_t0[head]) * n2;
        }
        P.counts[0] = nt;
        P.counts[1] = rows_total <= P.max_rows ? rows_total : P.max_rows;
        P.counts[2] = ni <= P.max_items ? ni : P.max_items;
    }
    __syncthreads();
    for (int g = tid; g < G; g += nthr) {
        // the member's gate/up tiles and its down tiles at their queue bases
        int j = sh_i0[g];
        for (int t = sh_t0[g]; t < sh_t0[g + 1]; ++t)
            for (int n = 0; n < n1; ++n, ++j)
                if (j < P.max_items) P.items[j] = make_int2(t, n);
        j = sh_d0[g];
        for (int t = sh_t0[g]; t < sh_t0[g + 1]; ++t)
            for (int n = 0; n < n2; ++n, ++j)
                if (j < P.max_items) P.items[j] = make_int2(t, 0x10000 | n);
        P.landed[g] = (sh_wp[g] & 1) ? 0u : nchunk;  // a hit is ready at once
    }
    for (int t = tid; t < nt; t += nthr) P.gu_done[t] = 0;
    for (int i0 = tid; i0 < nent; i0 += kAlignBatch * nthr) {
        int ew[kAlignBatch], id[kAlignBatch];
        load_entries(L, i0, nthr, nent, ew, id);
#pragma unroll
        for (int u = 0; u < kAlignBatch; ++u)
            if (ew[u] >= 0) {
                const int g = sh_g_of_e[id[u]];
                if (g < 0) continue;
                const int row = sh_off[g] + atomicAdd(&sh_fill[g], 1);
                if (row < P.max_rows) P.perm[row] = i0 + u * nthr;
            }
    }
    // padding rows: one warp per member
    const int lane = tid & 31;
    for (int g = tid >> 5; g < G; g += nthr >> 5) {
        const int cg = sh_cnt[g], padded = (cg + BM - 1) / BM * BM;
        for (int r = cg + lane; r < padded; r += 32)
            if (sh_off[g] + r < P.max_rows) P.perm[sh_off[g] + r] = -1;
    }
}

// ---------------------------------------------------------------- gather

// x_perm[r] = x[perm[r] / k] (zeros for padding rows): one warp per row.
__global__ void __launch_bounds__(256) prefill_gather_kernel(const __nv_bfloat16* __restrict__ x, PrefillDev P, int H,
                                                             int k) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int total = P.counts[1];
    const int nvec = H / 8;
    for (int r = blockIdx.x * 8 + (threadIdx.x >> 5); r < total; r += gridDim.x * 8) {
        const int e = P.perm[r];
        int4* dst = reinterpret_cast<int4*>(P.x_perm + (size_t)r * H);
        if (e >= 0) {
            const int4* src = reinterpret_cast<const int4*>(x + (size_t)(e / k) * H);
            for (int v = lane; v < nvec; v += 32) dst[v] = __ldg(src + v);
        } else {
            for (int v = lane; v < nvec; v += 32) dst[v] = make_int4(0, 0, 0, 0);
        }
    }
}

// ---------------------------------------------------------------- link role

// One 64 KiB item (a multiple of 16 bytes, possibly shorter at the row end).
__device__ __forceinline__ void link_copy(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, size_t bytes) {
    const int4* sp = reinterpret_cast<const int4*>(src);
    int4* dp = reinterpret_cast<int4*>(dst);
    const int nvec = (int)(bytes >> 4);
    int4 v[kLinkUnroll];
#pragma unroll
    for (int u = 0; u < kLinkUnroll; ++u) {
        const int i = threadIdx.x + u * kStepThreads;
        if (i < nvec) v[u] = ld_nc_na(sp + i);
    }
#pragma unroll
    for (int u = 0; u < kLinkUnroll; ++u) {
        const int i = threadIdx.x + u * kStepThreads;
        if (i < nvec) dp[i] = v[u];
    }
}

// A copy of `bytes` (a multiple of 16, at most kLinkChunk) within HBM,
// between rows written in this kernel: read through L2.
__device__ __forceinline__ void hbm_copy(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, size_t bytes) {
    const int4* sp = reinterpret_cast<const int4*>(src);
    int4* dp = reinterpret_cast<int4*>(dst);
    const int nvec = (int)(bytes >> 4);
    int4 v[kLinkUnroll];
#pragma unroll
    for (int u = 0; u < kLinkUnroll; ++u) {
        const int i = threadIdx.x + u * kStepThreads;
        if (i < nvec) v[u] = __ldcg(sp + i);
    }
#pragma unroll
    for (int u = 0; u < kLinkUnroll; ++u) {
        const int i = threadIdx.x + u * kStepThreads;
        if (i < nvec) dp[i] = v[u];
    }
}

// Link CTA `rank` of `nL`: items (page-in p, chunk c) in plan order, round
// robin, so the experts land one after another.  A page-in whose slot is
// still in use goes to its staging row if it has one, else it waits until
// the slot's earlier occupants' tiles are done.  Then the commit items copy
// each staged last occupant from its staging row into its slot, once the
// slot is free.
__device__ void link_role(const PrefillDev& P, const Shape& s, const uint8_t* __restrict__ host_layer,
                          uint8_t* __restrict__ slots_layer, uint8_t* __restrict__ slots_all, int rank, int nL,
                          unsigned nchunk, uint32_t* err, int* ok_sh) {
    const int np = P.counts[4], ncommit = P.counts[5];
    const size_t nstream = (size_t)np * nchunk, total = nstream + (size_t)ncommit * nchunk;
    int last_p = -1, last_ci = -1, ok = 1;
    for (size_t it = rank; it < total; it += nL) {
        if (it < nstream) {
            const int p = (int)(it / nchunk);
            const size_t c = it - (size_t)p * nchunk;
            const int g = P.pin_member[p];
            const int4 m = P.members[g];
            const int st = P.stage_of[g];
            if (p != last_p) {  // without a staging row the slot's earlier occupants must be done with it
                last_p = p;
                if (st < 0) {
                    if (threadIdx.x == 0)
                        *ok_sh = spin_geq(&P.slot_done[m.y], (unsigned)P.slot_need[g], &P.ctl[1], err);
                    __syncthreads();
                    ok = *ok_sh;
                } else {
                    ok = 1;
                }
            }
            const size_t off = c * kLinkChunk;
            uint8_t* row = st >= 0 ? slots_all + (size_t)(P.stage_base + st) * s.stride
                                   : slots_layer + (size_t)m.y * s.stride;
            if (ok) {
                const size_t n = s.copy_bytes - off < kLinkChunk ? s.copy_bytes - off : kLinkChunk;
                link_copy(host_layer + (size_t)m.x * s.stride + off, row + off, n);
            }
            __syncthreads();
            if (threadIdx.x == 0) {
                __threadfence();
                atomicAdd(&P.landed[g], 1u);
            }
        } else {
            const int ci = (int)((it - nstream) / nchunk);
            const size_t c = (it - nstream) - (size_t)ci * nchunk;
            const int g = P.commit_member[ci];
            const int4 m = P.members[g];
            const int st = P.stage_of[g];
            if (ci != last_ci) {  // the staging row has landed and the slot is free
                last_ci = ci;
                if (threadIdx.x == 0)
                    *ok_sh = spin_geq(&P.landed[g], nchunk, &P.ctl[1], err) &&
                             spin_geq(&P.slot_done[m.y], (unsigned)P.slot_need[g], &P.ctl[1], err);
                __syncthreads();
                ok = *ok_sh;
            }
            const size_t off = c * kLinkChunk;
            if (ok && st >= 0 && st < P.stage_rows) {
                const size_t n = s.copy_bytes - off < kLinkChunk ? s.copy_bytes - off : kLinkChunk;
                hbm_copy(slots_all + (size_t)(P.stage_base + st) * s.stride + off,
                         slots_layer + (size_t)m.y * s.stride + off, n);
            }
            __syncthreads();
        }
    }
}

// ---------------------------------------------------------------- GEMM role

// One GEMM tile as the scheduler hands it to the other roles.
struct TileInfo {
    int4 ti;    // row0, slot (whole table), valid rows, member
    int t;      // tile index (gate/up counters)
    int n;      // column tile
    int kind;   // 0 gate/up, 1 down, -1 no more tiles
    int ok;     // 0: a dependency wait gave up; the tile is skipped but counted
};

struct StepShared {
    uint64_t full[STAGES], empty[STAGES], conv[STAGES];
    uint64_t acc_full[2], acc_empty[2];
    uint64_t info_full[kInfoDepth], info_empty[kInfoDepth];
    TileInfo info[kInfoDepth];
    uint32_t tmem_base;
};

// A quantised tile's rows of the B operand for column tile n: gate rows
// n*BN/2.. and up rows I + n*BN/2.. (gate/up), or rows n*BN.. (down).
template <int EPI>
__device__ __forceinline__ int b_row(const Shape& s, int n_tile, int r) {
    return EPI == 0 ? (r < kQBN / 2 ? n_tile * (kQBN / 2) + r : s.I + n_tile * (kQBN / 2) + r - kQBN / 2)
                    : n_tile * kQBN + r;
}

// Producer: TMA loads of one tile's k-steps into the ring.
template <int EPI, int FMT>
__device__ __forceinline__ void produce_tile(const CUtensorMap* tmA, const CUtensorMap* tmB, StepShared& S,
                                             uint8_t* ring, const TileInfo& I, int kblocks, uint32_t kb0,
                                             const Shape& s, uint32_t* err) {
    constexpr bool QUANT = FMT != PE_BF16;
    constexpr int BN = Tile<FMT>::BN, AP = Tile<FMT>::A_PARTS;
    const bool two = I.ti.z > BM;  // only tiles of two A parts have more than 128 rows
    const int b_tx = QUANT ? Tile<FMT>::C_BYTES : Tile<FMT>::B_BYTES;
    for (int kb = 0; kb < kblocks; ++kb) {
        const uint32_t pos = kb0 + kb, st = pos % STAGES, use = pos / STAGES;
        if (use > 0 && !tc::mbar_wait(&S.empty[st], (use - 1) & 1, err, PE_DEVERR_TIMEOUT)) return;
        tc::mbar_arrive_expect_tx(&S.full[st], (two ? 2 * A_BYTES : A_BYTES) + b_tx);
        uint8_t* a = ring + st * Tile<FMT>::STAGE_BYTES;
        // bf16: the B tile itself; quantised: its codes, into the staging buffer
        uint8_t* b = QUANT ? a + AP * A_BYTES + Tile<FMT>::B_BYTES : a + AP * A_BYTES;
        // the weight map's inner coordinate counts bytes for int4 (two codes each)
        const int kx = is_4bit(FMT) ? kb * (BK / 2) : kb * BK;
        tc::tma_load_2d(a, tmA, &S.full[st], kb * BK, I.ti.x);
        if (two) tc::tma_load_2d(a + A_BYTES, tmA, &S.full[st], kb * BK, I.ti.x + BM);
        if (EPI == 0) {
            tc::tma_load_3d(b, tmB, &S.full[st], kx, I.n * (BN / 2), I.ti.y);
            tc::tma_load_3d(b + b_tx / 2, tmB, &S.full[st], kx, s.I + I.n * (BN / 2), I.ti.y);
        } else {
            tc::tma_load_3d(b, tmB, &S.full[st], kx, I.n * BN, I.ti.y);
        }
    }
}

// Converters (warps 2..11): decode the tile's weight codes into the
// swizzled bf16 B tile of each stage, applying the scales.
template <int EPI, int FMT>
__device__ __forceinline__ void convert_tile(StepShared& S, uint8_t* ring, float* scale, __half* scale4,
                                             const TileInfo& I, int kblocks, uint32_t kb0, const Shape& s,
                                             const uint8_t* slots_all, uint32_t* err) {
    constexpr int NCT = kConvWarps * 32;
    const int ct = threadIdx.x - 64, lane = threadIdx.x & 31;
    const int Kdim = EPI == 0 ? s.H : s.I;
    const int ng = Kdim / 128;  // FP8 block columns, int4 groups
    // the scales live in the slot, which this kernel's link CTAs write: read them through L2
    const uint8_t* sc = slots_all + (size_t)I.ti.y * s.stride + (EPI == 0 ? s.s13_off : s.s2_off);
    // every converter warp is done with the previous tile's scales
    asm volatile("bar.sync 1, %0;" ::"n"(NCT) : "memory");
    if (FMT == PE_FP8_BLOCK128) {
        // the tile's rows lie in one 128-row block per range (gate and up, or down)
        const int rb0 = b_row<EPI>(s, I.n, 0) / kFp8Block, rb1 = b_row<EPI>(s, I.n, kQBN - 1) / kFp8Block;
        for (int i = ct; i < 2 * ng; i += NCT) {
            const int h = i / ng, c = i - h * ng;
            scale[h * kMaxScaleCols + c] = __ldcg(reinterpret_cast<const float*>(sc) + (size_t)(h ? rb1 : rb0) * ng + c);
        }
    } else {
        // every row has its own scales (int4: [rows][K/128] fp16; MXFP4 /
        // NVFP4: [rows][K/32 or K/16] bytes after the grid's header); the
        // tile's rows are one or two contiguous 16-byte-aligned ranges: copy
        // as vectors
        const int row_bytes = FMT == PE_INT4_GPTQ ? ng * 2 : Kdim / fp4_block(FMT);
        const uint8_t* grid = sc + fp4_scale_header(FMT);
        const int half_vecs = (kQBN / 2) * row_bytes / 16;
        const uint8_t* src0 = grid + (size_t)b_row<EPI>(s, I.n, 0) * row_bytes;
        const uint8_t* src1 = grid + (size_t)b_row<EPI>(s, I.n, kQBN / 2) * row_bytes;
        int4* dst = reinterpret_cast<int4*>(scale4);
        for (int i = ct; i < 2 * half_vecs; i += NCT) {
            const uint8_t* src = i < half_vecs ? src0 + 16 * (size_t)i : src1 + 16 * (size_t)(i - half_vecs);
            dst[i] = __ldcg(reinterpret_cast<const int4*>(src));
        }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(NCT) : "memory");  // converter warps only
    for (int kb = 0; kb < kblocks; ++kb) {
        const uint32_t pos = kb0 + kb, st = pos % STAGES, use = pos / STAGES;
        if (!tc::mbar_wait(&S.full[st], use & 1, err, PE_DEVERR_TIMEOUT)) return;
        uint8_t* bt = ring + st * Tile<FMT>::STAGE_BYTES + Tile<FMT>::A_PARTS * A_BYTES;
        const uint8_t* codes = bt + Tile<FMT>::B_BYTES;
        for (int q = ct; q < kQBN * (BK / 16); q += NCT) {  // 16-code chunks: row r, chunk j
            const int r = q >> 2, j = q & 3;
            uint32_t packed[8];
            if (FMT == PE_FP8_BLOCK128) {
                const float scl = scale[((EPI == 0 && r >= kQBN / 2) ? kMaxScaleCols : 0) + (kb * BK) / kFp8Block];
                const int4 cv = *reinterpret_cast<const int4*>(codes + r * BK + j * 16);
                const uint32_t w4[4] = {(uint32_t)cv.x, (uint32_t)cv.y, (uint32_t)cv.z, (uint32_t)cv.w};
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const float2 lo = e4m3x2(w4[t]), hi = e4m3x2(w4[t] >> 16);
                    const __nv_bfloat162 p0 = __floats2bfloat162_rn(lo.x * scl, lo.y * scl);
                    const __nv_bfloat162 p1 = __floats2bfloat162_rn(hi.x * scl, hi.y * scl);
                    packed[2 * t] = *reinterpret_cast<const uint32_t*>(&p0);
                    packed[2 * t + 1] = *reinterpret_cast<const uint32_t*>(&p1);
                }
            } else if (FMT == PE_MXFP4 || FMT == PE_NVFP4) {
                // 2*e2m1(q) (exact bf16 pairs) times half the block scale, one
                // packed bf16 multiply.  Every product is exact: an E8M0 half is
                // a power of two, and 2*e2m1 (two significant bits) times an
                // E4M3 half (four) fits bf16's eight.  NVFP4's tensor scale is
                // applied to the fp32 accumulators in the epilogue.
                const int k0 = kb * BK + j * 16;
                const uint8_t* srow = reinterpret_cast<const uint8_t*>(scale4) + r * (Kdim / fp4_block(FMT));
                const float scl = FMT == PE_NVFP4 ? e4m3x2(srow[k0 / kNvfp4Block]).x * 0.5f
                                                  : e8m0_half(srow[k0 / kMxfp4Block]);
                const __nv_bfloat162 s2 = __float2bfloat162_rn(scl);
                const uint2 cv = *reinterpret_cast<const uint2*>(codes + r * (BK / 2) + j * 8);
#pragma unroll
                for (int h = 0; h < 2; ++h) {  // codes 8h .. 8h+7 of the chunk: one word
                    uint32_t p[4];
                    e2m1x8_bf16x2(h ? cv.y : cv.x, p);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const __nv_bfloat162 c2 = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&p[i]), s2);
                        packed[4 * h + i] = *reinterpret_cast<const uint32_t*>(&c2);
                    }
                }
            } else {
                // the fp16 scale's bits; each weight is the exact product (q - 8) * s rounded to bf16
                const uint32_t s16 = reinterpret_cast<const unsigned short*>(scale4)[r * ng + (kb * BK) / kInt4Group];
                const uint2 cv = *reinterpret_cast<const uint2*>(codes + r * (BK / 2) + j * 8);
#pragma unroll
                for (int h = 0; h < 2; ++h) {  // codes 8h .. 8h+7 of the chunk: one word
                    const uint32_t w = h ? cv.y : cv.x;
                    // q - 8 exactly, two codes at a time: nibbles (0,4), (1,5), (2,6), (3,7)
                    const uint32_t p04 = i4_pair_f16(w), p15 = i4_pair_f16(w >> 4);
                    const uint32_t p26 = i4_pair_f16(w >> 8), p37 = i4_pair_f16(w >> 12);
                    const __nv_bfloat162 c01 = __floats2bfloat162_rn(i4_lo_times(p04, s16), i4_lo_times(p15, s16));
                    const __nv_bfloat162 c23 = __floats2bfloat162_rn(i4_lo_times(p26, s16), i4_lo_times(p37, s16));
                    const __nv_bfloat162 c45 = __floats2bfloat162_rn(i4_hi_times(p04, s16), i4_hi_times(p15, s16));
                    const __nv_bfloat162 c67 = __floats2bfloat162_rn(i4_hi_times(p26, s16), i4_hi_times(p37, s16));
                    packed[4 * h] = *reinterpret_cast<const uint32_t*>(&c01);
                    packed[4 * h + 1] = *reinterpret_cast<const uint32_t*>(&c23);
                    packed[4 * h + 2] = *reinterpret_cast<const uint32_t*>(&c45);
                    packed[4 * h + 3] = *reinterpret_cast<const uint32_t*>(&c67);
                }
            }
            // bf16 columns 16j..16j+15 are the 16-byte chunks 2j, 2j+1 of row r, swizzled by r % 8
            uint8_t* row = bt + r * 128;
            *reinterpret_cast<int4*>(row + (((2 * j) ^ (r & 7)) * 16)) =
                make_int4(packed[0], packed[1], packed[2], packed[3]);
            *reinterpret_cast<int4*>(row + (((2 * j + 1) ^ (r & 7)) * 16)) =
                make_int4(packed[4], packed[5], packed[6], packed[7]);
        }
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&S.conv[st]);
    }
}

// MMA issuer: one tile into TMEM accumulator buffer acc (256 columns: one
// or two 128-row parts x BN).
template <int FMT>
__device__ __forceinline__ void mma_tile(StepShared& S, uint8_t* ring, const TileInfo& I, int kblocks, uint32_t kb0,
                                         uint32_t dst, uint32_t* err) {
    constexpr bool QUANT = FMT != PE_BF16;
    constexpr int BN = Tile<FMT>::BN;
    constexpr uint32_t idesc = tc::idesc_bf16_f32(BM, BN);
    const bool two = I.ti.z > BM;
    for (int kb = 0; kb < kblocks; ++kb) {
        const uint32_t pos = kb0 + kb, st = pos % STAGES, use = pos / STAGES;
        if (!tc::mbar_wait(QUANT ? &S.conv[st] : &S.full[st], use & 1, err, PE_DEVERR_TIMEOUT)) break;
        tc::fence_after_sync();
        const uint32_t a = tc::smem_u32(ring + st * Tile<FMT>::STAGE_BYTES);
        const uint32_t b = a + Tile<FMT>::A_PARTS * A_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t bd = tc::smem_desc_sw128(b + kk * 32);
            tc::mma_f16(dst, tc::smem_desc_sw128(a + kk * 32), bd, idesc, (kb | kk) != 0);
            if (two) tc::mma_f16(dst + BN, tc::smem_desc_sw128(a + A_BYTES + kk * 32), bd, idesc, (kb | kk) != 0);
        }
        tc::mma_commit(&S.empty[st]);  // frees the stage once these MMAs are done
    }
}

// SiLU for the prefill epilogue: the hardware exp2-based exponential and a
// fast divide (relative error around 1e-7, far inside the tolerances).  Paged
// and unpaged steps run this same code, so they still agree bit for bit.
__device__ __forceinline__ float silu_fast(float g) { return __fdividef(g, 1.f + __expf(-g)); }

// Epilogue (warps 12..15): warp w reads TMEM lanes 32*(w%4).. of the
// accumulator buffer; in row half hf, lane l owns tile row hf*128 + 32*(w%4) + l.
// TS: the accumulators are first multiplied by the weight tensor's scale ts
// (NVFP4, whose converters leave it out).
template <int EPI, int BN, bool TS>
__device__ __forceinline__ void epilogue_tile(const TileInfo& I, uint32_t acc, const PrefillDev& P, const LayerDev& L,
                                              const Shape& s, float ts, float* __restrict__ merged) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, quarter = warp & 3;
    for (int hf = 0; hf < (I.ti.z > BM ? 2 : 1); ++hf) {
        const int r = hf * BM + quarter * 32 + lane;
        const uint32_t trow = acc + hf * BN + ((uint32_t)(quarter * 32) << 16);
        if (EPI == 0) {
            for (int cc = 0; cc < BN / 64; ++cc) {  // 32 gate columns and the 32 up columns BN/2 further
                uint32_t g[32], u[32];
                tc::tmem_ld32(trow + cc * 32, g);
                tc::tmem_ld32(trow + BN / 2 + cc * 32, u);
                tc::tmem_ld_wait();
                if (r < I.ti.z) {
                    uint32_t packed[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        float g0 = __uint_as_float(g[2 * c]), g1 = __uint_as_float(g[2 * c + 1]);
                        float u0 = __uint_as_float(u[2 * c]), u1 = __uint_as_float(u[2 * c + 1]);
                        if (TS) {
                            g0 = __fmul_rn(ts, g0), g1 = __fmul_rn(ts, g1);
                            u0 = __fmul_rn(ts, u0), u1 = __fmul_rn(ts, u1);
                        }
                        const float h0 = __fmul_rn(silu_fast(g0), u0);
                        const float h1 = __fmul_rn(silu_fast(g1), u1);
                        const __nv_bfloat162 hv = __floats2bfloat162_rn(h0, h1);
                        packed[c] = *reinterpret_cast<const uint32_t*>(&hv);
                    }
                    int4* dst =
                        reinterpret_cast<int4*>(P.h_perm + (size_t)(I.ti.x + r) * s.I + I.n * (BN / 2) + cc * 32);
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        dst[v] = make_int4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
                }
            }
        } else {
            const int entry = r < I.ti.z ? P.perm[I.ti.x + r] : -1;
            const float w = entry >= 0 ? (TS ? __fmul_rn(L.topk_w[entry], ts) : L.topk_w[entry]) : 0.f;
            for (int c4 = 0; c4 < BN / 32; ++c4) {
                uint32_t v[32];
                tc::tmem_ld32(trow + c4 * 32, v);
                tc::tmem_ld_wait();
                if (entry >= 0) {
                    float4* dst = reinterpret_cast<float4*>(merged + (size_t)entry * s.H + I.n * BN + c4 * 32);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        dst[q] = make_float4(__fmul_rn(w, __uint_as_float(v[4 * q])),
                                             __fmul_rn(w, __uint_as_float(v[4 * q + 1])),
                                             __fmul_rn(w, __uint_as_float(v[4 * q + 2])),
                                             __fmul_rn(w, __uint_as_float(v[4 * q + 3])));
                }
            }
        }
    }
}

// ---------------------------------------------------------------- step kernel

template <int FMT>
__global__ void __launch_bounds__(kStepThreads, 1)
    prefill_step_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmH,
                        const __grid_constant__ CUtensorMap tmW13, const __grid_constant__ CUtensorMap tmW2,
                        PrefillDev P, LayerDev L, Shape s, const uint8_t* __restrict__ host_layer,
                        uint8_t* __restrict__ slots_all, int slot_base, int n1, int n2, unsigned nchunk,
                        float* __restrict__ merged, uint32_t* err) {
    constexpr bool QUANT = FMT != PE_BF16;
    extern __shared__ uint8_t smem_raw[];
    __shared__ StepShared S;
    __shared__ float sh_scale[FMT == PE_FP8_BLOCK128 ? 2 * kMaxScaleCols : 1];
    __shared__ __align__(16) __half sh_scale4[is_4bit(FMT) ? kScaleStageBytes / 2 : 8];
    __shared__ int sh_ok, sh_rank, sh_nlink;
    pdl_wait();
    // Roles follow the SM (every kLinkEvery-th SM streams the link), so they
    // stay spread over the GPU wherever the CTAs were placed.  Each CTA takes
    // a rank in its role; the link CTAs need their number.
    if (threadIdx.x == 0) {
        unsigned smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        const bool link = smid % kLinkEvery == 0;
        int rank = (int)atomicAdd(&P.ctl[link ? 2 : 3], 1u);
        int nlink = 0;
        bool all = false;
        for (uint32_t i = 0; i < kSpin && !all; ++i) {  // every CTA of the grid is resident: registration ends
            all = ld_acquire(&P.ctl[2]) + ld_acquire(&P.ctl[3]) >= gridDim.x;
            if (!all) __nanosleep(64);
        }
        if (!all) {
            // CTAs could read different link-CTA counts and split the page-ins
            // inconsistently: record the cause and abort the step, so every
            // wait gives up at once and the kernel ends
            atomicOr(err, PE_DEVERR_TIMEOUT);
            atomicExch(&P.ctl[1], 1u);
        }
        nlink = (int)ld_acquire(&P.ctl[2]);
        if (nlink == 0 && !link && rank == 0) {  // no SM of the link's kind: the first GEMM CTA streams it
            nlink = 1;
            rank = 0;
            sh_rank = 0;
        } else {
            sh_rank = link ? rank : -1;
        }
        sh_nlink = nlink == 0 ? 1 : nlink;
    }
    __syncthreads();
    if (sh_rank >= 0) {
        // a link CTA joins the GEMM queue once its share of the page-ins is
        // done (it then depends only on work queued before its next tile)
        link_role(P, s, host_layer, slots_all + (size_t)slot_base * s.stride, slots_all, sh_rank, sh_nlink, nchunk, err,
                  &sh_ok);
        __syncthreads();
    }

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    // readers of each tile-info entry: the MMA warp, the converter warps, the epilogue warps
    constexpr uint32_t kReaders = 1 + (QUANT ? kConvWarps : 0) + kEpiWarps;
    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            tc::mbar_init(&S.full[i], 1);
            tc::mbar_init(&S.empty[i], 1);
            tc::mbar_init(&S.conv[i], kConvWarps);  // one arrive per converter warp
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&S.acc_full[i], 1);
            tc::mbar_init(&S.acc_empty[i], kEpiWarps);
        }
        for (int i = 0; i < kInfoDepth; ++i) {
            tc::mbar_init(&S.info_full[i], 1);
            tc::mbar_init(&S.info_empty[i], kReaders);
        }
        tc::fence_barrier_init();
        tc::tma_prefetch(&tmX);
        tc::tma_prefetch(&tmH);
        tc::tma_prefetch(&tmW13);
        tc::tma_prefetch(&tmW2);
    }
    if (warp == 0) tc::tmem_alloc(&S.tmem_base, kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = S.tmem_base;
    const int nitems = P.counts[2];

    if (warp == 0) {
        // scheduler and TMA producer (lane 0): take a tile, wait for what it
        // reads, publish it to the other roles, stream its k-steps
        if (lane == 0) {
            uint32_t kb_ring = 0;
            for (uint32_t q = 0;; ++q) {
                const int j = (int)atomicAdd(&P.ctl[0], 1u);
                TileInfo I{make_int4(0, 0, 0, 0), 0, 0, -1, 0};
                if (j < nitems) {
                    const int2 it = P.items[j];
                    I.t = it.x;
                    I.kind = it.y >> 16;
                    I.n = it.y & 0xffff;
                    I.ti = P.tiles[it.x];
                    I.ok = I.kind == 0 ? spin_geq(&P.landed[I.ti.w], nchunk, &P.ctl[1], err)  // the expert has landed
                                       : spin_geq(&P.gu_done[it.x], (unsigned)n1, &P.ctl[1], err);  // its h is done
                    // the tensor-memory-access loads below read what other CTAs wrote
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                }
                const uint32_t e = q % kInfoDepth, use = q / kInfoDepth;
                if (use > 0) tc::mbar_wait(&S.info_empty[e], (use - 1) & 1, err, PE_DEVERR_TIMEOUT);
                S.info[e] = I;
                tc::mbar_arrive(&S.info_full[e]);
                if (I.kind < 0) break;
                if (!I.ok) continue;
                if (I.kind == 0) {
                    produce_tile<0, FMT>(&tmX, &tmW13, S, ring, I, s.H / BK, kb_ring, s, err);
                    kb_ring += s.H / BK;
                } else {
                    produce_tile<1, FMT>(&tmH, &tmW2, S, ring, I, s.I / BK, kb_ring, s, err);
                    kb_ring += s.I / BK;
                }
            }
        }
    } else if (warp == 1 || (QUANT && warp < 2 + kConvWarps) || warp >= 2 + kConvWarps) {
        const bool is_mma = warp == 1, is_conv = warp >= 2 && warp < 2 + kConvWarps;
        uint32_t kb_ring = 0, acc_iter = 0;
        for (uint32_t q = 0;; ++q) {
            const uint32_t e = q % kInfoDepth, use = q / kInfoDepth;
            tc::mbar_wait(&S.info_full[e], use & 1, err, PE_DEVERR_TIMEOUT);
            const TileInfo I = S.info[e];
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&S.info_empty[e]);
            if (I.kind < 0) break;
            const int kblocks = I.kind == 0 ? s.H / BK : s.I / BK;
            const uint32_t buf = acc_iter & 1, buse = acc_iter >> 1;
            if (I.ok) {
                if (is_mma) {
                    if (lane == 0) {
                        if (buse > 0) tc::mbar_wait(&S.acc_empty[buf], (buse - 1) & 1, err, PE_DEVERR_TIMEOUT);
                        tc::fence_after_sync();
                        mma_tile<FMT>(S, ring, I, kblocks, kb_ring, tmem + buf * kAccCols, err);
                        tc::mma_commit(&S.acc_full[buf]);
                    }
                    __syncwarp();
                } else if (is_conv) {
                    if (I.kind == 0)
                        convert_tile<0, FMT>(S, ring, sh_scale, sh_scale4, I, kblocks, kb_ring, s, slots_all, err);
                    else
                        convert_tile<1, FMT>(S, ring, sh_scale, sh_scale4, I, kblocks, kb_ring, s, slots_all, err);
                } else {  // epilogue
                    tc::mbar_wait(&S.acc_full[buf], buse & 1, err, PE_DEVERR_TIMEOUT);
                    tc::fence_after_sync();
                    constexpr bool TS = FMT == PE_NVFP4;
                    // NVFP4: the tensor scale from the head of the slot's scale grid
                    // (written with the codes, so present once they were converted)
                    const float ts =
                        TS ? __ldcg(reinterpret_cast<const float*>(slots_all + (size_t)I.ti.y * s.stride +
                                                                   (I.kind == 0 ? s.s13_off : s.s2_off)))
                           : 1.f;
                    if (I.kind == 0)
                        epilogue_tile<0, Tile<FMT>::BN, TS>(I, tmem + buf * kAccCols, P, L, s, ts, merged);
                    else
                        epilogue_tile<1, Tile<FMT>::BN, TS>(I, tmem + buf * kAccCols, P, L, s, ts, merged);
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(&S.acc_empty[buf]);  // the buffer may be overwritten
                }
                kb_ring += kblocks;
                ++acc_iter;
            }
            if (!is_mma && !is_conv) {
                // the tile's outputs are written (or it was skipped): count it
                asm volatile("bar.sync 2, %0;" ::"n"(kEpiWarps * 32) : "memory");
                if (warp == 2 + kConvWarps && lane == 0) {
                    __threadfence();
                    if (I.kind == 0) atomicAdd(&P.gu_done[I.t], 1u);
                    // tiles that read the slot itself (not a staging row)
                    if (I.ti.y < P.stage_base) atomicAdd(&P.slot_done[I.ti.y - slot_base], 1u);
                }
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
    // The next kernel is released only now: launched early, its CTAs were
    // measured to slow this multi-millisecond step down by about 10 %.
    pdl_trigger();
}

// Self-tests: a counter wait on a word nothing sets, and an mbarrier wait on
// a barrier nobody arrives on, must give up (and the counter wait must raise
// the abort word, after which a second wait gives up at once).
__global__ void prefill_wait_selftest_kernel(const unsigned* never, unsigned* abort_w, uint32_t* err_counter,
                                             uint32_t* err_mbar, uint32_t limit) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        spin_geq(never, 1u, abort_w, err_counter, limit);
        spin_geq(never, 1u, abort_w, err_counter, 4 * limit);  // the abort word ends it at once
        tc::mbar_init(&bar, 1);
        tc::fence_barrier_init();
        tc::mbar_wait(&bar, 0, err_mbar, PE_DEVERR_TIMEOUT, limit);
    }
}

int step_n1(const Shape& s) { return s.I / (prefill_bn(s.dtype) / 2); }
int step_n2(const Shape& s) { return s.H / prefill_bn(s.dtype); }
unsigned step_nchunk(const Shape& s) { return (unsigned)((s.copy_bytes + kLinkChunk - 1) / kLinkChunk); }
size_t align_smem(const Shape& s) { return sizeof(int) * ((size_t)2 * s.Wmax + (size_t)3 * s.Wmax * s.K); }
constexpr size_t kAlignMaxSmem = 160 * 1024;  // dynamic shared memory the align kernel may use

}  // namespace

bool prefill_tc_supported(const Shape& s) {
    if (s.dtype != PE_BF16 && s.dtype != PE_FP8_BLOCK128 && !is_4bit(s.dtype)) return false;
    if (align_smem(s) > kAlignMaxSmem) return false;
    if (s.dtype != PE_BF16 && (s.H > kMaxScaleCols * 128 || s.I > kMaxScaleCols * 128)) return false;
    // MXFP4 / NVFP4: a tile's scale rows (K / block bytes each) fit the staging buffer
    if ((s.dtype == PE_MXFP4 || s.dtype == PE_NVFP4) &&
        kQBN * (s.H > s.I ? s.H : s.I) / fp4_block(s.dtype) > kScaleStageBytes)
        return false;
    const int bn = prefill_bn(s.dtype);
    return s.H % bn == 0 && s.I % (bn / 2) == 0 && s.H % BK == 0 && s.I % BK == 0;
}

size_t prefill_max_rows(int max_entries, int E) {
    // every member is padded to a multiple of 128 rows; at most min(E, entries) members
    const size_t members = (size_t)(max_entries < E ? max_entries : E);
    const size_t rows = (size_t)max_entries + members * (BM - 1);
    return (rows + BM - 1) / BM * BM;
}

size_t prefill_max_tiles(int max_entries, int E) { return prefill_max_rows(max_entries, E) / BM; }

size_t prefill_max_items(const Shape& s, size_t max_tiles) { return max_tiles * (size_t)(step_n1(s) + step_n2(s)); }

cudaError_t prefill_setup_kernels() {
    cudaError_t e = cudaFuncSetAttribute(prefill_align_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kAlignMaxSmem);
    if (!e) e = cudaFuncSetAttribute(prefill_step_kernel<PE_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Tile<PE_BF16>::SMEM);
    if (!e)
        e = cudaFuncSetAttribute(prefill_step_kernel<PE_FP8_BLOCK128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Tile<PE_FP8_BLOCK128>::SMEM);
    if (!e)
        e = cudaFuncSetAttribute(prefill_step_kernel<PE_INT4_GPTQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Tile<PE_INT4_GPTQ>::SMEM);
    if (!e)
        e = cudaFuncSetAttribute(prefill_step_kernel<PE_MXFP4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Tile<PE_MXFP4>::SMEM);
    if (!e)
        e = cudaFuncSetAttribute(prefill_step_kernel<PE_NVFP4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Tile<PE_NVFP4>::SMEM);
    return e;
}

cudaError_t prefill_step_ctas_per_sm(int dtype, int* out) {
    int n = 0;
    cudaError_t e = dtype == PE_FP8_BLOCK128
                        ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, prefill_step_kernel<PE_FP8_BLOCK128>,
                                                                        kStepThreads, Tile<PE_FP8_BLOCK128>::SMEM)
                    : dtype == PE_INT4_GPTQ
                        ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, prefill_step_kernel<PE_INT4_GPTQ>,
                                                                        kStepThreads, Tile<PE_INT4_GPTQ>::SMEM)
                    : dtype == PE_MXFP4
                        ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, prefill_step_kernel<PE_MXFP4>,
                                                                        kStepThreads, Tile<PE_MXFP4>::SMEM)
                    : dtype == PE_NVFP4
                        ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, prefill_step_kernel<PE_NVFP4>,
                                                                        kStepThreads, Tile<PE_NVFP4>::SMEM)
                        : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, prefill_step_kernel<PE_BF16>, kStepThreads,
                                                                        Tile<PE_BF16>::SMEM);
    *out = e ? 0 : n;
    return e;
}

cudaError_t selftest_prefill_waits(const unsigned* never, unsigned* abort_w, uint32_t* err_counter,
                                   uint32_t* err_mbar, uint32_t limit, cudaStream_t st) {
    prefill_wait_selftest_kernel<<<1, 32, 0, st>>>(never, abort_w, err_counter, err_mbar, limit);
    return cudaGetLastError();
}

cudaError_t launch_prefill_align(const LayerDev& L, const Shape& s, const PrefillDev& P, const __nv_bfloat16* x,
                                 int slot_base, int T, int num_sms, cudaStream_t st) {
    // down tiles trail their gate/up tiles by two rounds of the GEMM CTAs
    const int gemm_ctas = num_sms - (num_sms + kLinkEvery - 1) / kLinkEvery;
    cudaError_t e = launch_pdl(prefill_align_kernel, 1, 1024, align_smem(s), st, L, s, P, slot_base, T, step_n1(s),
                               step_n2(s), step_nchunk(s), 2 * (gemm_ctas > 1 ? gemm_ctas : 1),
                               prefill_mt(s.dtype));
    if (e) return e;
    return launch_pdl(prefill_gather_kernel, num_sms * 4, 256, 0, st, x, P, s.H, s.k);
}

cudaError_t launch_prefill_step(const LayerDev& L, const Shape& s, const PrefillDev& P, const PrefillMaps& M,
                                const uint8_t* host_layer, uint8_t* slots_all, int slot_base, float* merged,
                                uint32_t* err, int num_sms, cudaStream_t st) {
    const int grid = num_sms < kLinkEvery + 1 ? kLinkEvery + 1 : num_sms;  // at least one CTA of each role
    const int n1 = step_n1(s), n2 = step_n2(s);
    const unsigned nchunk = step_nchunk(s);
#define PE_STEP(F)                                                                                          \
    return launch_pdl(prefill_step_kernel<F>, grid, kStepThreads, Tile<F>::SMEM, st, M.x_perm, M.h_perm, M.w13, M.w2, \
                      P, L, s, host_layer, slots_all, slot_base, n1, n2, nchunk, merged, err)
    if (s.dtype == PE_FP8_BLOCK128) PE_STEP(PE_FP8_BLOCK128);
    if (s.dtype == PE_INT4_GPTQ) PE_STEP(PE_INT4_GPTQ);
    if (s.dtype == PE_MXFP4) PE_STEP(PE_MXFP4);
    if (s.dtype == PE_NVFP4) PE_STEP(PE_NVFP4);
    PE_STEP(PE_BF16);
#undef PE_STEP
}

}  // namespace pe
