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
// Every row of an MMA tile is computed independently and always with the same
// k order, so an entry's result does not depend on its tile-mates, its slot
// or its wave: paged and unpaged prefill agree bit for bit.

#include "pe_device.cuh"
#include "pe_internal.h"
#include "tc_sm100.cuh"

namespace pe {
namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 3;
constexpr int MT = 2 * BM;                   // rows of one tile: two M=128 MMAs
constexpr int A_BYTES = BM * BK * 2;         // one 128-row half of the A tile
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = 2 * A_BYTES + B_BYTES;
constexpr int GEMM_SMEM = STAGES * STAGE_BYTES + 1024;  // + slack to align the ring to 1024 B
constexpr uint32_t kTmemCols = 2 * BN;       // one 128-column accumulator per half

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
template <int EPI>
__global__ void __launch_bounds__(128, 1) prefill_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                                                              const __grid_constant__ CUtensorMap tmB, PrefillDev P,
                                                              LayerDev L, Shape s, int n_tiles, int kblocks,
                                                              float* __restrict__ merged, uint32_t* err) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[STAGES];
    __shared__ __align__(8) uint64_t empty_bar[STAGES];
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
            tc::mbar_arrive_expect_tx(&full_bar[st], two ? STAGE_BYTES : STAGE_BYTES - A_BYTES);
            uint8_t* a = ring + st * STAGE_BYTES;
            uint8_t* b = a + 2 * A_BYTES;
            tc::tma_load_2d(a, &tmA, &full_bar[st], kb * BK, ti.x);
            if (two) tc::tma_load_2d(a + A_BYTES, &tmA, &full_bar[st], kb * BK, ti.x + BM);
            if (EPI == 0) {
                tc::tma_load_3d(b, &tmB, &full_bar[st], kb * BK, n_tile * (BN / 2), ti.y);
                tc::tma_load_3d(b + B_BYTES / 2, &tmB, &full_bar[st], kb * BK, s.I + n_tile * (BN / 2), ti.y);
            } else {
                tc::tma_load_3d(b, &tmB, &full_bar[st], kb * BK, n_tile * BN, ti.y);
            }
        }
    } else if (warp == 1 && lane == 0) {  // MMA issuer
        constexpr uint32_t idesc = tc::idesc_bf16_f32(BM, BN);
        for (int kb = 0; kb < kblocks; ++kb) {
            const int st = kb % STAGES, use = kb / STAGES;
            if (!tc::mbar_wait(&full_bar[st], use & 1, err, PE_DEVERR_TIMEOUT)) break;
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
    return s.dtype == PE_BF16 && s.H % BN == 0 && s.I % (BN / 2) == 0 && s.H % BK == 0 && s.I % BK == 0;
}

size_t prefill_max_rows(int max_entries, int K) {
    const size_t rows = (size_t)max_entries + (size_t)K * (BM - 1);
    return (rows + BM - 1) / BM * BM;
}

cudaError_t prefill_setup_kernels() {
    cudaError_t e = cudaFuncSetAttribute(prefill_gemm_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM);
    if (!e) e = cudaFuncSetAttribute(prefill_gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM);
    return e;
}

cudaError_t launch_prefill_align(const LayerDev& L, const Shape& s, const PrefillDev& P, const __nv_bfloat16* x,
                                 int slot_base, int wave, int T, int num_sms, cudaStream_t st) {
    cudaError_t e = launch_pdl(prefill_align_kernel, 1, 1024, 0, st, L, s, P, slot_base, wave, T);
    if (e) return e;
    return launch_pdl(prefill_gather_kernel, num_sms * 4, 256, 0, st, x, P, s.H, s.k);
}

cudaError_t launch_prefill_gemm(int which, const LayerDev& L, const Shape& s, const PrefillDev& P,
                                const PrefillMaps& M, float* merged, uint32_t* err, cudaStream_t st) {
    const int m_tiles = P.max_tiles;
    if (which == 0) {
        const int n1 = s.I / (BN / 2);
        return launch_pdl(prefill_gemm_kernel<0>, m_tiles * n1, 128, (size_t)GEMM_SMEM, st, M.x_perm, M.w13, P, L, s,
                          n1, s.H / BK, merged, err);
    }
    const int n2 = s.H / BN;
    return launch_pdl(prefill_gemm_kernel<1>, m_tiles * n2, 128, (size_t)GEMM_SMEM, st, M.h_perm, M.w2, P, L, s, n2,
                      s.I / BK, merged, err);
}

}  // namespace pe
