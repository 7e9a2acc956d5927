// Prefill-sized expert MLP on the tcgen05 tensor cores.
//
// "Paged Experts" (SGLang docs), "A step: waves, page-in, merge", step 3: the
// fused-MoE kernel runs over the wave's own entries, without its top-k sum,
// each output already multiplied by its router weight.  At prefill sizes an
// expert has tens to hundreds of routed tokens, so its MLP is a pair of dense
// contractions:
//   GEMM1: [rows_e, H] x w13[2I, H]^T  -> SiLU(gate) * up -> h [rows_e, I] (bf16)
//   GEMM2: [rows_e, I] x w2[H, I]^T    -> * router weight -> merged entries (fp32)
//
// Per wave:
//   align   one CTA groups the wave's entries by member expert, pads every
//           member to a multiple of 128 rows and writes the row -> entry map
//           and a tile table (row offset, slot, valid rows);
//   gather  copies each entry's token row of x into the packed A operand;
//   GEMM1/2 one CTA per (up to 256 rows of one expert) x 256 output columns:
//           TMA (128-byte swizzle) feeds a 3-stage shared-memory ring, one
//           thread issues two M=128 tcgen05.mma per k-step that share the
//           weight tile (the second only when the expert has more than 128
//           rows), the accumulators live in TMEM, and four warps run the
//           epilogue from TMEM.  Each weight slice is read once per 256 rows.
// The weights come straight from the slot table (a 3-D tensor map over
// [slot][row][k]), so a page-in is all it takes to make them visible.
//
// Block-FP8 experts (E4M3 codes, one fp32 scale per 128x128 block) keep bf16
// activations: TMA brings the code tile into a staging buffer, two converter
// warps decode it, multiply by its block scale, round to bf16 and write it in
// the 128-byte-swizzled layout the MMA reads; the MMA then runs as for bf16.
//
// Every row of an MMA tile is computed independently and always with the same
// k order, so an entry's result does not depend on its tile-mates, its slot
// or its wave: paged and unpaged prefill agree bit for bit.

#include "fp8_device.cuh"
#include "pe_device.cuh"
#include "pe_internal.h"
#include "tc_sm100.cuh"

namespace pe {
namespace {

constexpr int BM = 128, BK = 64, STAGES = 3;
constexpr int MT = 2 * BM;            // rows of one tile: two M=128 MMAs
constexpr int A_BYTES = BM * BK * 2;  // one 128-row half of the A tile

// Tile geometry per weight format.  Stage layout: [A half 0][A half 1]
// [B tile, bf16, swizzled][FP8 only: code staging], every part 1024-aligned.
template <bool FP8>
struct Tile {
    static constexpr int BN = FP8 ? 128 : 256;       // output columns (MMA N)
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int C_BYTES = FP8 ? BN * BK : 0;  // E4M3 codes of the B tile
    static constexpr int STAGE_BYTES = 2 * A_BYTES + B_BYTES + C_BYTES;
    static constexpr int SMEM = STAGES * STAGE_BYTES + 1024;  // + slack to align the ring
    static constexpr uint32_t TMEM_COLS = 2 * BN;    // one accumulator per 128-row half
};

// ---------------------------------------------------------------- align

__global__ void __launch_bounds__(1024) prefill_align_kernel(LayerDev L, Shape s, PrefillDev P, int slot_base,
                                                             int wave, int T) {
    __shared__ int sh_cnt[kMaxSlots], sh_off[kMaxSlots], sh_fill[kMaxSlots], sh_q_of_slot[kMaxSlots];
    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int size = L.member_count[wave];
    const int nent = T * s.k;
    for (int i = tid; i < s.K; i += nthr) sh_q_of_slot[i] = -1;
    for (int q = tid; q < size; q += nthr) {
        sh_cnt[q] = 0;
        sh_fill[q] = 0;
    }
    __syncthreads();
    for (int q = tid; q < size; q += nthr) sh_q_of_slot[L.member_slot[(size_t)wave * s.K + q]] = q;
    __syncthreads();
    for (int i = tid; i < nent; i += nthr)
        if (L.entry_wave[i] == wave) {
            const int q = sh_q_of_slot[L.entry_slot[i]];
            if (q >= 0) atomicAdd(&sh_cnt[q], 1);
        }
    __syncthreads();
    if (tid == 0) {
        int off = 0, nt = 0;
        for (int q = 0; q < size; ++q) {
            sh_off[q] = off;
            const int c = sh_cnt[q];
            const int slot = L.member_slot[(size_t)wave * s.K + q];
            for (int r = 0; r < c && nt < P.max_tiles; r += MT)
                P.tiles[nt++] = make_int4(off + r, slot_base + slot, min(MT, c - r), q);
            off += (c + BM - 1) / BM * BM;
        }
        P.counts[0] = nt;
        P.counts[1] = off <= P.max_rows ? off : P.max_rows;
    }
    __syncthreads();
    for (int i = tid; i < nent; i += nthr)
        if (L.entry_wave[i] == wave) {
            const int q = sh_q_of_slot[L.entry_slot[i]];
            if (q < 0) continue;
            const int row = sh_off[q] + atomicAdd(&sh_fill[q], 1);
            if (row < P.max_rows) P.perm[row] = i;
        }
    for (int q = 0; q < size; ++q) {
        const int c = sh_cnt[q], padded = (c + BM - 1) / BM * BM;
        for (int r = c + tid; r < padded; r += nthr)
            if (sh_off[q] + r < P.max_rows) P.perm[sh_off[q] + r] = -1;
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

// ---------------------------------------------------------------- GEMM

// EPI 0: A = x_perm, B = w13 (gate rows n0.. and up rows I+n0.., 128 each),
//        h_perm[row, n0 + c] = bf16(SiLU(gate_c) * up_c), c < 128.
// EPI 1: A = h_perm, B = w2 rows m0..m0+255,
//        merged[entry, m0 + c] = w_entry * acc_c.
template <int EPI, bool FP8>
__global__ void __launch_bounds__(128, 1) prefill_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                                                              const __grid_constant__ CUtensorMap tmB, PrefillDev P,
                                                              LayerDev L, Shape s, const uint8_t* __restrict__ slots_all,
                                                              int n_tiles, int kblocks, float* __restrict__ merged,
                                                              uint32_t* err) {
    using TL = Tile<FP8>;
    constexpr int BN = TL::BN, B_BYTES = TL::B_BYTES, STAGE_BYTES = TL::STAGE_BYTES;
    constexpr uint32_t kTmemCols = TL::TMEM_COLS;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[STAGES];
    __shared__ __align__(8) uint64_t empty_bar[STAGES];
    __shared__ __align__(8) uint64_t conv_bar[STAGES];  // FP8: the bf16 B tile is written
    __shared__ __align__(8) uint64_t acc_bar;
    __shared__ uint32_t tmem_base_sh;
    pdl_wait();
    pdl_trigger();
    const int m_tile = blockIdx.x / n_tiles, n_tile = blockIdx.x - (blockIdx.x / n_tiles) * n_tiles;
    if (m_tile >= P.counts[0]) return;  // uniform per CTA: nothing allocated yet
    const int4 ti = P.tiles[m_tile];     // row0, slot (global), valid rows, member
    const bool two = ti.z > BM;          // the tile's second 128-row half is used
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            tc::mbar_init(&full_bar[i], 1);
            tc::mbar_init(&empty_bar[i], 1);
            tc::mbar_init(&conv_bar[i], 2);  // one arrive per converter warp
        }
        tc::mbar_init(&acc_bar, 1);
        tc::fence_barrier_init();
        tc::tma_prefetch(&tmA);
        tc::tma_prefetch(&tmB);
    }
    if (warp == 0) tc::tmem_alloc(&tmem_base_sh, kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_base_sh;

    if (warp == 0 && lane == 0) {  // TMA producer
        for (int kb = 0; kb < kblocks; ++kb) {
            const int st = kb % STAGES, use = kb / STAGES;
            if (use > 0 && !tc::mbar_wait(&empty_bar[st], (use - 1) & 1, err, PE_DEVERR_TIMEOUT)) break;
            const int b_tx = FP8 ? TL::C_BYTES : B_BYTES;
            tc::mbar_arrive_expect_tx(&full_bar[st], (two ? 2 * A_BYTES : A_BYTES) + b_tx);
            uint8_t* a = ring + st * STAGE_BYTES;
            // bf16: the B tile itself; FP8: its codes, into the staging buffer
            uint8_t* b = FP8 ? a + 2 * A_BYTES + B_BYTES : a + 2 * A_BYTES;
            tc::tma_load_2d(a, &tmA, &full_bar[st], kb * BK, ti.x);
            if (two) tc::tma_load_2d(a + A_BYTES, &tmA, &full_bar[st], kb * BK, ti.x + BM);
            if (EPI == 0) {
                tc::tma_load_3d(b, &tmB, &full_bar[st], kb * BK, n_tile * (BN / 2), ti.y);
                tc::tma_load_3d(b + b_tx / 2, &tmB, &full_bar[st], kb * BK, s.I + n_tile * (BN / 2), ti.y);
            } else {
                tc::tma_load_3d(b, &tmB, &full_bar[st], kb * BK, n_tile * BN, ti.y);
            }
        }
    } else if (warp == 1 && lane == 0) {  // MMA issuer
        constexpr uint32_t idesc = tc::idesc_bf16_f32(BM, BN);
        for (int kb = 0; kb < kblocks; ++kb) {
            const int st = kb % STAGES, use = kb / STAGES;
            if (!tc::mbar_wait(FP8 ? &conv_bar[st] : &full_bar[st], use & 1, err, PE_DEVERR_TIMEOUT)) break;
            tc::fence_after_sync();
            const uint32_t a = tc::smem_u32(ring + st * STAGE_BYTES);
            const uint32_t b = a + 2 * A_BYTES;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
                const uint64_t bd = tc::smem_desc_sw128(b + kk * 32);
                tc::mma_f16(tmem, tc::smem_desc_sw128(a + kk * 32), bd, idesc, (kb | kk) != 0);
                if (two) tc::mma_f16(tmem + BN, tc::smem_desc_sw128(a + A_BYTES + kk * 32), bd, idesc, (kb | kk) != 0);
            }
            tc::mma_commit(&empty_bar[st]);  // frees the stage once these MMAs are done
        }
        tc::mma_commit(&acc_bar);
    } else if (FP8 && warp >= 2) {  // converters: E4M3 codes -> scaled bf16, swizzled
        const int ct = threadIdx.x - 64;
        const int Kdim = EPI == 0 ? s.H : s.I;
        const int nbk = (Kdim + kFp8Block - 1) / kFp8Block;
        const float* sc = reinterpret_cast<const float*>(slots_all + (size_t)ti.y * s.stride + (EPI == 0 ? s.s13_off : s.s2_off));
        for (int kb = 0; kb < kblocks; ++kb) {
            const int st = kb % STAGES, use = kb / STAGES;
            if (!tc::mbar_wait(&full_bar[st], use & 1, err, PE_DEVERR_TIMEOUT)) break;
            uint8_t* bt = ring + st * STAGE_BYTES + 2 * A_BYTES;
            const uint8_t* codes = bt + B_BYTES;
            for (int q = ct; q < BN * (BK / 16); q += 64) {  // 16-code chunks: row r, chunk j
                const int r = q >> 2, j = q & 3;
                const int grow = EPI == 0 ? (r < BN / 2 ? n_tile * (BN / 2) + r : s.I + n_tile * (BN / 2) + r - BN / 2)
                                          : n_tile * BN + r;
                const float scale = __ldg(sc + (size_t)(grow / kFp8Block) * nbk + (kb * BK) / kFp8Block);
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
                *reinterpret_cast<int4*>(row + (((2 * j) ^ (r & 7)) * 16)) = make_int4(packed[0], packed[1], packed[2], packed[3]);
                *reinterpret_cast<int4*>(row + (((2 * j + 1) ^ (r & 7)) * 16)) = make_int4(packed[4], packed[5], packed[6], packed[7]);
            }
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&conv_bar[st]);
        }
    }
    __syncwarp();

    // epilogue: in half hf, thread r owns tile row hf*128 + r (TMEM lane r,
    // accumulator columns hf*128 ..)
    const bool ok = tc::mbar_wait(&acc_bar, 0, err, PE_DEVERR_TIMEOUT);
    tc::fence_after_sync();
    for (int hf = 0; hf < (two ? 2 : 1); ++hf) {
        const int r = hf * BM + warp * 32 + lane;
        const uint32_t trow = tmem + hf * BN + ((uint32_t)(warp * 32) << 16);
        if (EPI == 0) {
            for (int cc = 0; cc < BN / 64; ++cc) {  // 32-column chunks of gate (and up, BN/2 further)
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
                    int4* dst = reinterpret_cast<int4*>(P.h_perm + (size_t)(ti.x + r) * s.I + n_tile * (BN / 2) + cc * 32);
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        dst[v] = make_int4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
                }
            }
        } else {
            const int entry = r < ti.z ? P.perm[ti.x + r] : -1;
            const float w = entry >= 0 ? L.topk_w[entry] : 0.f;
            for (int c4 = 0; c4 < BN / 32; ++c4) {
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
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

bool prefill_tc_supported(const Shape& s) {
    if (s.dtype == PE_FP8_BLOCK128) {
        constexpr int BN = Tile<true>::BN;
        return s.H % BN == 0 && s.I % (BN / 2) == 0 && s.H % BK == 0 && s.I % BK == 0;
    }
    constexpr int BN = Tile<false>::BN;
    return s.dtype == PE_BF16 && s.H % BN == 0 && s.I % (BN / 2) == 0 && s.H % BK == 0 && s.I % BK == 0;
}

size_t prefill_max_rows(int max_entries, int K) {
    const size_t rows = (size_t)max_entries + (size_t)K * (BM - 1);
    return (rows + BM - 1) / BM * BM;
}

cudaError_t prefill_setup_kernels() {
    cudaError_t e = cudaFuncSetAttribute(prefill_gemm_kernel<0, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Tile<false>::SMEM);
    if (!e)
        e = cudaFuncSetAttribute(prefill_gemm_kernel<1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Tile<false>::SMEM);
    if (!e)
        e = cudaFuncSetAttribute(prefill_gemm_kernel<0, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Tile<true>::SMEM);
    if (!e)
        e = cudaFuncSetAttribute(prefill_gemm_kernel<1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Tile<true>::SMEM);
    return e;
}

cudaError_t launch_prefill_align(const LayerDev& L, const Shape& s, const PrefillDev& P, const __nv_bfloat16* x,
                                 int slot_base, int wave, int T, int num_sms, cudaStream_t st) {
    cudaError_t e = launch_pdl(prefill_align_kernel, 1, 1024, 0, st, L, s, P, slot_base, wave, T);
    if (e) return e;
    return launch_pdl(prefill_gather_kernel, num_sms * 4, 256, 0, st, x, P, s.H, s.k);
}

cudaError_t launch_prefill_gemm(int which, const LayerDev& L, const Shape& s, const PrefillDev& P,
                                const PrefillMaps& M, const uint8_t* slots_all, float* merged, uint32_t* err,
                                cudaStream_t st) {
    const int m_tiles = P.max_tiles;
    const bool fp8 = s.dtype == PE_FP8_BLOCK128;
    const int bn = fp8 ? Tile<true>::BN : Tile<false>::BN;
    const size_t smem = fp8 ? Tile<true>::SMEM : Tile<false>::SMEM;
    if (which == 0) {
        const int n1 = s.I / (bn / 2);
        return fp8 ? launch_pdl(prefill_gemm_kernel<0, true>, m_tiles * n1, 128, smem, st, M.x_perm, M.w13, P, L, s,
                                slots_all, n1, s.H / BK, merged, err)
                   : launch_pdl(prefill_gemm_kernel<0, false>, m_tiles * n1, 128, smem, st, M.x_perm, M.w13, P, L, s,
                                slots_all, n1, s.H / BK, merged, err);
    }
    const int n2 = s.H / bn;
    return fp8 ? launch_pdl(prefill_gemm_kernel<1, true>, m_tiles * n2, 128, smem, st, M.h_perm, M.w2, P, L, s,
                            slots_all, n2, s.I / BK, merged, err)
               : launch_pdl(prefill_gemm_kernel<1, false>, m_tiles * n2, 128, smem, st, M.h_perm, M.w2, P, L, s,
                            slots_all, n2, s.I / BK, merged, err);
}

}  // namespace pe
