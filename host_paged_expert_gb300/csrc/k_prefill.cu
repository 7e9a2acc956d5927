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
//           table, the GEMM work queue, the page-in list, and for each
//           member how many GEMM tiles of its slot's earlier occupants in
//           this step must finish before its page-in may overwrite the slot;
//   gather  copies each entry's token row of x into the packed A operand;
//   step    one persistent CTA per SM.  Every fourth CTA streams the host
//           link: it copies 64 KiB chunks of the planned experts, in plan
//           order, from the pinned host store into their slots and counts
//           each expert's landed chunks.  The other CTAs take GEMM tiles
//           from a queue in the same order (the hits of wave 0 first): a
//           gate/up tile starts once every chunk of its expert has landed, a
//           down tile once all gate/up tiles of its rows are done.  So the
//           resident experts compute while the misses page in, every paged
//           expert computes as soon as it has landed, and wave w+1's page-in
//           runs under wave w's GEMMs, slot by slot.
// The waves stay exactly the planner's: a page-in never overwrites a slot
// before the GEMMs of the slot's previous expert are done with it.
//
// A GEMM tile is up to 256 rows of one expert x BN output columns.  TMA
// (128-byte swizzle) feeds a 3-stage shared-memory ring, one thread issues
// two M=128 tcgen05.mma per k-step that share the weight tile (the second
// only when the expert has more than 128 rows), the accumulators live in
// TMEM, and eight warps run the epilogue from TMEM.  The weights come straight
// from the slot table (a 3-D tensor map over [slot][row][k]).
//
// Block-FP8 experts (E4M3 codes, one fp32 scale per 128x128 block) and GPTQ
// int4 experts (4-bit codes, zero point 8, one fp16 scale per output row and
// 128 inputs) keep bf16 activations: TMA brings the code tile into a staging
// buffer, six converter warps decode it, multiply by its scale, round to bf16
// and write it in the 128-byte-swizzled layout the MMA reads; the MMA then
// runs as for bf16.  A tile's scales are staged in shared memory once per
// tile (FP8: one row of blocks for each of its gate, up or down row ranges;
// int4: every row's group scales).
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

#include "fp8_device.cuh"
#include "pe_device.cuh"
#include "pe_internal.h"
#include "tc_sm100.cuh"

namespace pe {
namespace {

constexpr int BM = 128, BK = 64, STAGES = 3;
constexpr int MT = 2 * BM;            // rows of one tile: two M=128 MMAs
constexpr int A_BYTES = BM * BK * 2;  // one 128-row half of the A tile
constexpr int kStepThreads = 256;
constexpr int kLinkEvery = 4;         // CTAs 0, 4, 8, ... of the step stream the host link
constexpr int kLinkUnroll = 16;
constexpr size_t kLinkChunk = (size_t)kStepThreads * 16 * kLinkUnroll;  // 64 KiB per item
constexpr int kConvWarps = 6;         // FP8 / int4: warps 2..7 decode the weight tiles
constexpr int kMaxScaleCols = 64;     // FP8 / int4: K / 128 of either GEMM (H, I <= 8192)
constexpr uint32_t kSpin = 1u << 22;  // polls, >= 128 ns apart

// Tile geometry per weight format (PE_BF16, PE_FP8_BLOCK128, PE_INT4_GPTQ).
// Stage layout: [A half 0][A half 1][B tile, bf16, swizzled][quantised
// formats only: code staging], every part 1024-aligned.
template <int FMT>
struct Tile {
    static constexpr int BN = FMT == PE_BF16 ? 256 : 128;  // output columns (MMA N)
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int C_BYTES = FMT == PE_FP8_BLOCK128 ? BN * BK          // E4M3 codes of the B tile
                                   : FMT == PE_INT4_GPTQ  ? BN * BK / 2      // int4 codes of the B tile
                                                          : 0;
    static constexpr int STAGE_BYTES = 2 * A_BYTES + B_BYTES + C_BYTES;
    static constexpr int SMEM = STAGES * STAGE_BYTES + 1024;  // + slack to align the ring
    static constexpr uint32_t TMEM_COLS = 2 * BN;      // one accumulator per 128-row half
};

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Thread-level bounded wait for *p >= target.  Gives up at once when the
// step's abort word is set; running out of polls records the timeout and
// sets the abort word.
__device__ __forceinline__ int spin_geq(const unsigned* p, unsigned target, unsigned* abort_w, uint32_t* err) {
    for (uint32_t i = 0; i < kSpin; ++i) {
        if (ld_acquire(p) >= target) return 1;
        if (*reinterpret_cast<volatile unsigned*>(abort_w)) return 0;
        __nanosleep(128);
    }
    atomicOr(err, PE_DEVERR_TIMEOUT);
    atomicExch(abort_w, 1u);
    return 0;
}

// ---------------------------------------------------------------- align

__global__ void __launch_bounds__(1024) prefill_align_kernel(LayerDev L, Shape s, PrefillDev P, int slot_base, int T,
                                                             int n1, int n2, unsigned nchunk) {
    __shared__ int sh_g_of_e[kMaxExperts];  // expert -> member
    __shared__ int sh_me[kMaxExperts], sh_ms[kMaxExperts], sh_paged[kMaxExperts];
    __shared__ int sh_cnt[kMaxExperts], sh_off[kMaxExperts], sh_fill[kMaxExperts];
    __shared__ int sh_t0[kMaxExperts + 1], sh_i0[kMaxExperts];
    __shared__ int sh_cum[kMaxSlots];
    __shared__ int sh_G;
    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int nent = T * s.k, K = s.K;
    for (int e = tid; e < s.E; e += nthr) sh_g_of_e[e] = -1;
    for (int i = tid; i < K; i += nthr) {
        sh_cum[i] = 0;
        P.slot_done[i] = 0;
    }
    if (tid == 0) {
        // members in queue order: wave by wave; in each wave the hits (no
        // page-in to wait for) first, then the page-ins in plan order
        const int nW = min(*L.num_waves, s.Wmax);
        int g = 0, np = 0;
        for (int w = 0; w < nW; ++w) {
            const int size = L.member_count[w], nmiss = L.plan_count[w];
            for (int pass = 0; pass < 2; ++pass) {
                const int q0 = pass == 0 ? nmiss : 0, q1 = pass == 0 ? size : nmiss;
                for (int q = q0; q < q1; ++q) {
                    const int e = L.member_expert[(size_t)w * K + q], slot = L.member_slot[(size_t)w * K + q];
                    sh_me[g] = e;
                    sh_ms[g] = slot;
                    sh_paged[g] = pass;
                    P.members[g] = make_int4(e, slot, w, pass);
                    if (pass) P.pin_member[np++] = g;
                    ++g;
                }
            }
        }
        sh_G = g;
        P.counts[3] = g;
        P.counts[4] = np;
        P.ctl[0] = 0;  // GEMM ticket
        P.ctl[1] = 0;  // abort word
    }
    __syncthreads();
    const int G = sh_G;
    for (int g = tid; g < G; g += nthr) {
        sh_g_of_e[sh_me[g]] = g;
        sh_cnt[g] = 0;
        sh_fill[g] = 0;
    }
    __syncthreads();
    for (int i = tid; i < nent; i += nthr)
        if (L.entry_wave[i] >= 0) {
            const int g = sh_g_of_e[L.topk_id[i]];
            if (g >= 0) atomicAdd(&sh_cnt[g], 1);
        }
    __syncthreads();
    if (tid == 0) {
        int off = 0, nt = 0, ni = 0;
        for (int g = 0; g < G; ++g) {
            const int c = sh_cnt[g], slot = sh_ms[g];
            sh_off[g] = off;
            sh_t0[g] = nt;
            for (int r = 0; r < c && nt < P.max_tiles; r += MT)
                P.tiles[nt++] = make_int4(off + r, slot_base + slot, min(MT, c - r), g);
            const int work = (nt - sh_t0[g]) * (n1 + n2);
            sh_i0[g] = ni;
            ni += work;
            // GEMM tiles of this slot's earlier occupants (members are in wave order)
            P.slot_need[g] = sh_cum[slot];
            sh_cum[slot] += work;
            off += (c + BM - 1) / BM * BM;
        }
        sh_t0[G] = nt;
        P.counts[0] = nt;
        P.counts[1] = off <= P.max_rows ? off : P.max_rows;
        P.counts[2] = ni <= P.max_items ? ni : P.max_items;
    }
    __syncthreads();
    for (int g = tid; g < G; g += nthr) {
        // the member's gate/up tiles, then its down tiles
        int j = sh_i0[g];
        for (int t = sh_t0[g]; t < sh_t0[g + 1]; ++t)
            for (int n = 0; n < n1; ++n, ++j)
                if (j < P.max_items) P.items[j] = make_int2(t, n);
        for (int t = sh_t0[g]; t < sh_t0[g + 1]; ++t)
            for (int n = 0; n < n2; ++n, ++j)
                if (j < P.max_items) P.items[j] = make_int2(t, 0x10000 | n);
        P.landed[g] = sh_paged[g] ? 0u : nchunk;  // a hit is ready at once
    }
    for (int t = tid; t < sh_t0[G]; t += nthr) P.gu_done[t] = 0;
    for (int i = tid; i < nent; i += nthr)
        if (L.entry_wave[i] >= 0) {
            const int g = sh_g_of_e[L.topk_id[i]];
            if (g < 0) continue;
            const int row = sh_off[g] + atomicAdd(&sh_fill[g], 1);
            if (row < P.max_rows) P.perm[row] = i;
        }
    for (int g = 0; g < G; ++g) {
        const int c = sh_cnt[g], padded = (c + BM - 1) / BM * BM;
        for (int r = c + tid; r < padded; r += nthr)
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

// Link CTA `rank` of `nL`: items (page-in p, chunk c) in plan order, round
// robin, so the experts land one after another.
__device__ void link_role(const PrefillDev& P, const Shape& s, const uint8_t* __restrict__ host_layer,
                          uint8_t* __restrict__ slots_layer, int rank, int nL, unsigned nchunk, uint32_t* err,
                          int* ok_sh) {
    const int np = P.counts[4];
    const size_t total = (size_t)np * nchunk;
    int last_p = -1, ok = 1;
    for (size_t it = rank; it < total; it += nL) {
        const int p = (int)(it / nchunk);
        const size_t c = it - (size_t)p * nchunk;
        const int g = P.pin_member[p];
        const int4 m = P.members[g];
        if (p != last_p) {  // the slot's earlier occupants in this step must be done with it
            last_p = p;
            if (threadIdx.x == 0) *ok_sh = spin_geq(&P.slot_done[m.y], (unsigned)P.slot_need[g], &P.ctl[1], err);
            __syncthreads();
            ok = *ok_sh;
        }
        const size_t off = c * kLinkChunk;
        if (ok) {
            const size_t n = s.copy_bytes - off < kLinkChunk ? s.copy_bytes - off : kLinkChunk;
            link_copy(host_layer + (size_t)m.x * s.stride + off, slots_layer + (size_t)m.y * s.stride + off, n);
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence();
            atomicAdd(&P.landed[g], 1u);
        }
    }
}

// ---------------------------------------------------------------- GEMM role

struct Ring {
    uint8_t* base;
    uint64_t* full;
    uint64_t* empty;
    uint64_t* conv;  // quantised formats: the bf16 B tile of the stage is written
    uint64_t* acc;
    float* scale;    // FP8: [2][kMaxScaleCols] block scales of the tile's two row ranges
    __half* scale4;  // int4: [BN][kMaxScaleCols] group scales of the tile's rows
};

// One tile.  EPI 0: A = x_perm, B = w13 (gate rows n0.. and up rows I+n0..,
//   BN/2 each), h_perm[row, n0 + c] = bf16(SiLU(gate_c) * up_c), c < BN/2.
// EPI 1: A = h_perm, B = w2 rows m0..m0+BN-1, merged[entry, m0 + c] = w * acc_c.
// kb0 = k-steps this CTA ran before (ring position); acc_phase = tiles before, mod 2.
template <int EPI, int FMT>
__device__ __forceinline__ void gemm_tile(const CUtensorMap* tmA, const CUtensorMap* tmB, const Ring& R, int4 ti,
                                          int n_tile, int kblocks, uint32_t kb0, uint32_t acc_phase, uint32_t tmem,
                                          const PrefillDev& P, const LayerDev& L, const Shape& s,
                                          const uint8_t* slots_all, float* __restrict__ merged, uint32_t* err) {
    using TL = Tile<FMT>;
    constexpr bool QUANT = FMT != PE_BF16;
    constexpr int BN = TL::BN, B_BYTES = TL::B_BYTES, STAGE_BYTES = TL::STAGE_BYTES;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool two = ti.z > BM;  // the tile's second 128-row half is used

    if (threadIdx.x == 0) {  // TMA producer
        for (int kb = 0; kb < kblocks; ++kb) {
            const uint32_t pos = kb0 + kb, st = pos % STAGES, use = pos / STAGES;
            if (use > 0 && !tc::mbar_wait(&R.empty[st], (use - 1) & 1, err, PE_DEVERR_TIMEOUT)) break;
            const int b_tx = QUANT ? TL::C_BYTES : B_BYTES;
            tc::mbar_arrive_expect_tx(&R.full[st], (two ? 2 * A_BYTES : A_BYTES) + b_tx);
            uint8_t* a = R.base + st * STAGE_BYTES;
            // bf16: the B tile itself; quantised: its codes, into the staging buffer
            uint8_t* b = QUANT ? a + 2 * A_BYTES + B_BYTES : a + 2 * A_BYTES;
            // the weight map's inner coordinate counts bytes for int4 (two codes each)
            const int kx = FMT == PE_INT4_GPTQ ? kb * (BK / 2) : kb * BK;
            tc::tma_load_2d(a, tmA, &R.full[st], kb * BK, ti.x);
            if (two) tc::tma_load_2d(a + A_BYTES, tmA, &R.full[st], kb * BK, ti.x + BM);
            if (EPI == 0) {
                tc::tma_load_3d(b, tmB, &R.full[st], kx, n_tile * (BN / 2), ti.y);
                tc::tma_load_3d(b + b_tx / 2, tmB, &R.full[st], kx, s.I + n_tile * (BN / 2), ti.y);
            } else {
                tc::tma_load_3d(b, tmB, &R.full[st], kx, n_tile * BN, ti.y);
            }
        }
    } else if (threadIdx.x == 32) {  // MMA issuer
        constexpr uint32_t idesc = tc::idesc_bf16_f32(BM, BN);
        for (int kb = 0; kb < kblocks; ++kb) {
            const uint32_t pos = kb0 + kb, st = pos % STAGES, use = pos / STAGES;
            if (!tc::mbar_wait(QUANT ? &R.conv[st] : &R.full[st], use & 1, err, PE_DEVERR_TIMEOUT)) break;
            tc::fence_after_sync();
            const uint32_t a = tc::smem_u32(R.base + st * STAGE_BYTES);
            const uint32_t b = a + 2 * A_BYTES;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
                const uint64_t bd = tc::smem_desc_sw128(b + kk * 32);
                tc::mma_f16(tmem, tc::smem_desc_sw128(a + kk * 32), bd, idesc, (kb | kk) != 0);
                if (two) tc::mma_f16(tmem + BN, tc::smem_desc_sw128(a + A_BYTES + kk * 32), bd, idesc, (kb | kk) != 0);
            }
            tc::mma_commit(&R.empty[st]);  // frees the stage once these MMAs are done
        }
        tc::mma_commit(R.acc);
    } else if (FMT == PE_INT4_GPTQ && warp >= 2) {  // converters: int4 codes -> scaled bf16, swizzled
        constexpr int NCT = kConvWarps * 32;
        const int ct = threadIdx.x - 64;
        const int Kdim = EPI == 0 ? s.H : s.I;
        const int ng = Kdim / kInt4Group;
        {
            // every row of the tile has its own group scales; they live in
            // the slot, which this kernel's link CTAs write: read through L2
            const unsigned short* sc = reinterpret_cast<const unsigned short*>(
                slots_all + (size_t)ti.y * s.stride + (EPI == 0 ? s.s13_off : s.s2_off));
            for (int i = ct; i < BN * ng; i += NCT) {
                const int r = i / ng, c = i - r * ng;
                const int grow = EPI == 0 ? (r < BN / 2 ? n_tile * (BN / 2) + r : s.I + n_tile * (BN / 2) + r - BN / 2)
                                          : n_tile * BN + r;
                R.scale4[r * kMaxScaleCols + c] = __ushort_as_half(__ldcg(sc + (size_t)grow * ng + c));
            }
            asm volatile("bar.sync 1, %0;" ::"n"(NCT) : "memory");  // converter warps only
        }
        for (int kb = 0; kb < kblocks; ++kb) {
            const uint32_t pos = kb0 + kb, st = pos % STAGES, use = pos / STAGES;
            if (!tc::mbar_wait(&R.full[st], use & 1, err, PE_DEVERR_TIMEOUT)) break;
            uint8_t* bt = R.base + st * STAGE_BYTES + 2 * A_BYTES;
            const uint8_t* codes = bt + B_BYTES;
            const int grp = (kb * BK) / kInt4Group;
            for (int q = ct; q < BN * (BK / 16); q += NCT) {  // 16-code chunks: row r, chunk j
                const int r = q >> 2, j = q & 3;
                const float scale = __half2float(R.scale4[r * kMaxScaleCols + grp]);
                const uint2 cv = *reinterpret_cast<const uint2*>(codes + r * (BK / 2) + j * 8);
                uint32_t packed[8];
#pragma unroll
                for (int t = 0; t < 8; ++t) {  // codes 2t, 2t+1 of the chunk
                    const uint32_t w = t < 4 ? cv.x : cv.y;
                    const int sh = 8 * (t & 3);
                    const float v0 = (float)(int)((w >> sh) & 0xFu) - 8.f;
                    const float v1 = (float)(int)((w >> (sh + 4)) & 0xFu) - 8.f;
                    const __nv_bfloat162 pv = __floats2bfloat162_rn(v0 * scale, v1 * scale);
                    packed[t] = *reinterpret_cast<const uint32_t*>(&pv);
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
            if (lane == 0) tc::mbar_arrive(&R.conv[st]);
        }
    } else if (FMT == PE_FP8_BLOCK128 && warp >= 2) {  // converters: E4M3 codes -> scaled bf16, swizzled
        constexpr int NCT = kConvWarps * 32;
        const int ct = threadIdx.x - 64;
        const int Kdim = EPI == 0 ? s.H : s.I;
        const int nbk = (Kdim + kFp8Block - 1) / kFp8Block;
        {
            // The tile's rows lie in one 128-row block per range (gate and up
            // for w13, one range for w2).  The scales live in the slot, which
            // this kernel's link CTAs write: read them through L2.
            const float* sc = reinterpret_cast<const float*>(slots_all + (size_t)ti.y * s.stride +
                                                             (EPI == 0 ? s.s13_off : s.s2_off));
            const int rb0 = EPI == 0 ? n_tile * (BN / 2) / kFp8Block : n_tile * BN / kFp8Block;
            const int rb1 = EPI == 0 ? (s.I + n_tile * (BN / 2)) / kFp8Block : rb0;
            for (int i = ct; i < 2 * nbk; i += NCT) {
                const int h = i / nbk, c = i - h * nbk;
                R.scale[h * kMaxScaleCols + c] = __ldcg(sc + (size_t)(h ? rb1 : rb0) * nbk + c);
            }
            asm volatile("bar.sync 1, %0;" ::"n"(NCT) : "memory");  // converter warps only
        }
        for (int kb = 0; kb < kblocks; ++kb) {
            const uint32_t pos = kb0 + kb, st = pos % STAGES, use = pos / STAGES;
            if (!tc::mbar_wait(&R.full[st], use & 1, err, PE_DEVERR_TIMEOUT)) break;
            uint8_t* bt = R.base + st * STAGE_BYTES + 2 * A_BYTES;
            const uint8_t* codes = bt + B_BYTES;
            const float* srow = R.scale + (kb * BK) / kFp8Block;
            for (int q = ct; q < BN * (BK / 16); q += NCT) {  // 16-code chunks: row r, chunk j
                const int r = q >> 2, j = q & 3;
                const float scale = srow[(EPI == 0 && r >= BN / 2) ? kMaxScaleCols : 0];
                const int4 cv = *reinterpret_cast<const int4*>(codes + r * BK + j * 16);
                const uint32_t w4[4] = {(uint32_t)cv.x, (uint32_t)cv.y, (uint32_t)cv.z, (uint32_t)cv.w};
                uint32_t packed[8];
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const float2 lo = e4m3x2(w4[t]), hi = e4m3x2(w4[t] >> 16);
                    const __nv_bfloat162 p0 = __floats2bfloat162_rn(lo.x * scale, lo.y * scale);
                    const __nv_bfloat162 p1 = __floats2bfloat162_rn(hi.x * scale, hi.y * scale);
                    packed[2 * t] = *reinterpret_cast<const uint32_t*>(&p0);
                    packed[2 * t + 1] = *reinterpret_cast<const uint32_t*>(&p1);
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
            if (lane == 0) tc::mbar_arrive(&R.conv[st]);
        }
    }
    __syncwarp();

    // epilogue: warp w reads TMEM lanes 32*(w%4).. (its lane quarter) and the
    // (w/4)-th half of the tile's output columns; in row half hf, lane l owns
    // tile row hf*128 + 32*(w%4) + l
    const bool ok = tc::mbar_wait(R.acc, acc_phase, err, PE_DEVERR_TIMEOUT);
    tc::fence_after_sync();
    const int quarter = warp & 3, colh = warp >> 2;
    for (int hf = 0; hf < (two ? 2 : 1); ++hf) {
        const int r = hf * BM + quarter * 32 + lane;
        const uint32_t trow = tmem + hf * BN + ((uint32_t)(quarter * 32) << 16);
        if (EPI == 0) {
            constexpr int NCH = BN / 128;  // 32-column chunks of gate (and up, BN/2 further) per column half
            for (int c0 = 0; c0 < NCH; ++c0) {
                const int cc = colh * NCH + c0;
                uint32_t g[32], u[32];
                tc::tmem_ld32(trow + cc * 32, g);
                tc::tmem_ld32(trow + BN / 2 + cc * 32, u);
                tc::tmem_ld_wait();
                if (ok && r < ti.z) {
                    uint32_t packed[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const float h0 = __fmul_rn(silu(__uint_as_float(g[2 * c])), __uint_as_float(u[2 * c]));
                        const float h1 = __fmul_rn(silu(__uint_as_float(g[2 * c + 1])), __uint_as_float(u[2 * c + 1]));
                        const __nv_bfloat162 hv = __floats2bfloat162_rn(h0, h1);
                        packed[c] = *reinterpret_cast<const uint32_t*>(&hv);
                    }
                    int4* dst =
                        reinterpret_cast<int4*>(P.h_perm + (size_t)(ti.x + r) * s.I + n_tile * (BN / 2) + cc * 32);
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        dst[v] = make_int4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
                }
            }
        } else {
            const int entry = r < ti.z ? P.perm[ti.x + r] : -1;
            const float w = entry >= 0 ? L.topk_w[entry] : 0.f;
            constexpr int NCH = BN / 64;  // 32-column chunks per column half
            for (int c0 = 0; c0 < NCH; ++c0) {
                const int c4 = colh * NCH + c0;
                uint32_t v[32];
                tc::tmem_ld32(trow + c4 * 32, v);
                tc::tmem_ld_wait();
                if (ok && entry >= 0) {
                    float4* dst = reinterpret_cast<float4*>(merged + (size_t)entry * s.H + n_tile * BN + c4 * 32);
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
    using TL = Tile<FMT>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[STAGES];
    __shared__ __align__(8) uint64_t empty_bar[STAGES];
    __shared__ __align__(8) uint64_t conv_bar[STAGES];
    __shared__ __align__(8) uint64_t acc_bar;
    __shared__ float sh_scale[FMT == PE_FP8_BLOCK128 ? 2 * kMaxScaleCols : 1];
    __shared__ __half sh_scale4[FMT == PE_INT4_GPTQ ? Tile<FMT>::BN * kMaxScaleCols : 1];
    __shared__ uint32_t tmem_base_sh;
    __shared__ int2 sh_item;
    __shared__ int sh_ok;
    pdl_wait();
    pdl_trigger();
    if (blockIdx.x % kLinkEvery == 0) {
        link_role(P, s, host_layer, slots_all + (size_t)slot_base * s.stride, blockIdx.x / kLinkEvery,
                  (gridDim.x + kLinkEvery - 1) / kLinkEvery, nchunk, err, &sh_ok);
        return;
    }

    const int warp = threadIdx.x >> 5;
    Ring R{reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023)), full_bar,
           empty_bar, conv_bar, &acc_bar, sh_scale, sh_scale4};
    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            tc::mbar_init(&full_bar[i], 1);
            tc::mbar_init(&empty_bar[i], 1);
            tc::mbar_init(&conv_bar[i], kConvWarps);  // one arrive per converter warp
        }
        tc::mbar_init(&acc_bar, 1);
        tc::fence_barrier_init();
        tc::tma_prefetch(&tmX);
        tc::tma_prefetch(&tmH);
        tc::tma_prefetch(&tmW13);
        tc::tma_prefetch(&tmW2);
    }
    if (warp == 0) tc::tmem_alloc(&tmem_base_sh, TL::TMEM_COLS);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_base_sh;
    const int nitems = P.counts[2];
    uint32_t kb_ring = 0, acc_phase = 0;
    for (;;) {
        if (threadIdx.x == 0) {
            const int j = (int)atomicAdd(&P.ctl[0], 1u);
            int2 it = make_int2(-1, 0);
            int ok = 0;
            if (j < nitems) {
                it = P.items[j];
                if ((it.y >> 16) == 0)  // gate/up: every chunk of the expert has landed
                    ok = spin_geq(&P.landed[P.tiles[it.x].w], nchunk, &P.ctl[1], err);
                else  // down: all gate/up tiles of these rows are done
                    ok = spin_geq(&P.gu_done[it.x], (unsigned)n1, &P.ctl[1], err);
                // the tensor-memory-access loads below read what other CTAs wrote
                asm volatile("fence.proxy.async.global;" ::: "memory");
            }
            sh_item = it;
            sh_ok = ok;
        }
        __syncthreads();
        tc::fence_after_sync();
        const int2 it = sh_item;
        if (it.x < 0) break;
        const bool down = (it.y >> 16) != 0;
        const int n = it.y & 0xffff;
        const int4 ti = P.tiles[it.x];
        if (sh_ok) {
            if (!down) {
                gemm_tile<0, FMT>(&tmX, &tmW13, R, ti, n, s.H / BK, kb_ring, acc_phase, tmem, P, L, s, slots_all,
                                  merged, err);
                kb_ring += s.H / BK;
            } else {
                gemm_tile<1, FMT>(&tmH, &tmW2, R, ti, n, s.I / BK, kb_ring, acc_phase, tmem, P, L, s, slots_all,
                                  merged, err);
                kb_ring += s.I / BK;
            }
            acc_phase ^= 1u;
        }
        tc::fence_before_sync();
        __syncthreads();  // the tile's outputs are written and its TMEM reads are done
        if (threadIdx.x == 0) {
            __threadfence();
            if (!down) atomicAdd(&P.gu_done[it.x], 1u);
            atomicAdd(&P.slot_done[ti.y - slot_base], 1u);
        }
    }
    if (warp == 0) tc::tmem_dealloc(tmem, TL::TMEM_COLS);
}

int step_bn(const Shape& s) { return s.dtype == PE_BF16 ? Tile<PE_BF16>::BN : Tile<PE_FP8_BLOCK128>::BN; }
int step_n1(const Shape& s) { return s.I / (step_bn(s) / 2); }
int step_n2(const Shape& s) { return s.H / step_bn(s); }
unsigned step_nchunk(const Shape& s) { return (unsigned)((s.copy_bytes + kLinkChunk - 1) / kLinkChunk); }

}  // namespace

bool prefill_tc_supported(const Shape& s) {
    if (s.dtype != PE_BF16 && s.dtype != PE_FP8_BLOCK128 && s.dtype != PE_INT4_GPTQ) return false;
    if (s.dtype != PE_BF16 && (s.H > kMaxScaleCols * 128 || s.I > kMaxScaleCols * 128)) return false;
    const int BN = step_bn(s);
    return s.H % BN == 0 && s.I % (BN / 2) == 0 && s.H % BK == 0 && s.I % BK == 0;
}

size_t prefill_max_rows(int max_entries, int E) {
    // every member is padded to a multiple of 128 rows; at most min(E, entries) members
    const size_t members = (size_t)(max_entries < E ? max_entries : E);
    const size_t rows = (size_t)max_entries + members * (BM - 1);
    return (rows + BM - 1) / BM * BM;
}

size_t prefill_max_items(const Shape& s, size_t max_tiles) { return max_tiles * (size_t)(step_n1(s) + step_n2(s)); }

cudaError_t prefill_setup_kernels() {
    cudaError_t e = cudaFuncSetAttribute(prefill_step_kernel<PE_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Tile<PE_BF16>::SMEM);
    if (!e)
        e = cudaFuncSetAttribute(prefill_step_kernel<PE_FP8_BLOCK128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Tile<PE_FP8_BLOCK128>::SMEM);
    if (!e)
        e = cudaFuncSetAttribute(prefill_step_kernel<PE_INT4_GPTQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Tile<PE_INT4_GPTQ>::SMEM);
    return e;
}

cudaError_t launch_prefill_align(const LayerDev& L, const Shape& s, const PrefillDev& P, const __nv_bfloat16* x,
                                 int slot_base, int T, int num_sms, cudaStream_t st) {
    cudaError_t e = launch_pdl(prefill_align_kernel, 1, 1024, 0, st, L, s, P, slot_base, T, step_n1(s), step_n2(s),
                               step_nchunk(s));
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
    PE_STEP(PE_BF16);
#undef PE_STEP
}

}  // namespace pe
