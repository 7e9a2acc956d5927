// Block-FP8 expert MLP for decode sizes ("Paged Experts", SGLang docs,
// "Supported Configurations and Limitations": block-quantised FP8 with a
// [128, 128] weight block).  Weights are E4M3 codes with one fp32 scale per
// 128x128 block: W[n, c] = e4m3(q[n, c]) * s[n / 128][c / 128].  Activations
// stay bf16 and accumulation is fp32.
//
// The kernels mirror the bf16 ones (k_gemv.cu): gate/up with the page-in
// fused in, the same on resident slots only, and the down projection with
// the top-k sum.  A 16-byte chunk holds 16 codes of one row and never crosses
// a 128-column block, so each lane decodes its chunk (hardware E4M3 -> f16,
// exact), forms the chunk's dot product and adds it scaled by the chunk's
// block scale.  Scales are read from the same place as the codes (host row
// for a page-in, slot for a hit), so a slot never pairs one expert's codes
// with another's scales.

#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "fp8_device.cuh"
#include "pe_device.cuh"
#include "pe_internal.h"

namespace pe {
namespace {

constexpr int kThreads8 = 256;
constexpr int kWarps8 = kThreads8 / 32;
constexpr int kCopyLoads8 = 8;
constexpr size_t kWarpCopy8 = (size_t)32 * 16 * kCopyLoads8;
constexpr int kDownRows8 = 8;
constexpr int kSmemBudget8 = 48 * 1024;

// Gate/up of one wave fused with its page-in; same work split as the bf16
// kernel (link CTAs: page-in rows used for h, then the rest of each paged row;
// HBM CTAs: resident members' rows).
template <int CPL>
__global__ void __launch_bounds__(kThreads8, 2) gateup_pagein_fp8_kernel(
    LayerDev L, Shape s, const __nv_bfloat16* __restrict__ x, const uint8_t* __restrict__ host,
    uint8_t* __restrict__ slots, int wave, int T, float* __restrict__ hbuf, int stage_x) {
    extern __shared__ int4 sh_dyn8[];
    int32_t* sh_mexp = reinterpret_cast<int32_t*>(sh_dyn8);
    int32_t* sh_mslot = sh_mexp + s.K;
    int32_t* sh_ekey = sh_mslot + s.K;
    const int nent = T * s.k;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    pdl_wait();
    pdl_trigger();
    const int size = L.member_count[wave];
    const int count = L.plan_count[wave];
    for (int i = threadIdx.x; i < size; i += blockDim.x) {
        sh_mexp[i] = L.member_expert[(size_t)wave * s.K + i];
        sh_mslot[i] = L.member_slot[(size_t)wave * s.K + i];
    }
    for (int i = threadIdx.x; i < nent; i += blockDim.x)
        sh_ekey[i] = L.entry_wave[i] == wave ? L.entry_slot[i] : -1;
    const uint8_t* xbase = reinterpret_cast<const uint8_t*>(x);
    if (stage_x) {
        int4* sx = reinterpret_cast<int4*>(sh_mexp + ((2 * s.K + nent + 3) & ~3));
        const int nvec = T * s.H / 8;
        for (int i = threadIdx.x; i < nvec; i += blockDim.x) sx[i] = ldg16(xbase + 16 * (size_t)i);
        xbase = reinterpret_cast<const uint8_t*>(sx);
    }
    __syncthreads();

    const int nchunk = s.H >> 4;
    const size_t xrow = (size_t)s.H * 2;
    const long long miss_rows = (long long)count * s.I;
    const size_t tail_bytes = s.copy_bytes - s.tail_off;
    const long long copies_per = (long long)((tail_bytes + kWarpCopy8 - 1) / kWarpCopy8);
    const long long link_items = miss_rows + (long long)count * copies_per;
    const long long hbm_items = (long long)(size - count) * s.I;
    const int G = gridDim.x;
    const int Gl = link_items == 0 ? 0 : hbm_items == 0 ? G : max(1, G / 2);
    const bool link_cta = (int)blockIdx.x < Gl;
    const long long first = (long long)(link_cta ? blockIdx.x : blockIdx.x - Gl) * kWarps8 + warp;
    const long long stride = (long long)(link_cta ? Gl : G - Gl) * kWarps8;
    const long long total = link_cta ? link_items : hbm_items;
    for (long long item = first; item < total; item += stride) {
        if (link_cta && item >= miss_rows) {
            const long long c = item - miss_rows;
            const int q = (int)(c / copies_per);
            const size_t off = s.tail_off + (size_t)(c - (long long)q * copies_per) * kWarpCopy8;
            const uint8_t* src = host + (size_t)sh_mexp[q] * s.stride + off;
            uint8_t* dst = slots + (size_t)sh_mslot[q] * s.stride + off;
            const size_t nbytes = min(kWarpCopy8, s.copy_bytes - off);
            int4 v[kCopyLoads8];
#pragma unroll
            for (int u = 0; u < kCopyLoads8; ++u) {
                const size_t o = ((size_t)u * 32 + lane) * 16;
                if (o < nbytes) v[u] = ld_nc_na(src + o);
            }
#pragma unroll
            for (int u = 0; u < kCopyLoads8; ++u) {
                const size_t o = ((size_t)u * 32 + lane) * 16;
                if (o < nbytes) *reinterpret_cast<int4*>(dst + o) = v[u];
            }
            continue;
        }
        const int q = link_cta ? (int)(item / s.I) : count + (int)(item / s.I);
        const int n = (int)(item % s.I);
        const int slot = sh_mslot[q];
        uint8_t* slot_base = slots + (size_t)slot * s.stride;
        const uint8_t* base = link_cta ? host + (size_t)sh_mexp[q] * s.stride : slot_base;
        int4 gv[CPL], uv[CPL];
        float sg[CPL], su[CPL];
        load_row_pair_fp8<CPL>(base, s, n, lane, nchunk, link_cta, gv, uv, sg, su);
        if (link_cta) {
            uint8_t* gd = slot_base + s.w13_off + (size_t)n * s.H;
            uint8_t* ud = gd + (size_t)s.I * s.H;
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
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
                const float h = row_pair_h_fp8<CPL>(gv, uv, sg, su, xbase + (size_t)(ei / s.k) * xrow, lane, nchunk);
                if (lane == 0) hbuf[(size_t)ei * s.I + n] = h;
            }
        }
    }
}

// Gate/up of one wave from the slots only (after a separate page-in): one
// warp per (entry, row).
template <int CPL>
__global__ void __launch_bounds__(kThreads8) gateup_fp8_kernel(LayerDev L, Shape s, const __nv_bfloat16* __restrict__ x,
                                                              const uint8_t* __restrict__ slots, int wave, int T,
                                                              float* __restrict__ hbuf) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int nchunk = s.H >> 4;
    const long long total = (long long)T * s.k * s.I;
    for (long long item = (long long)blockIdx.x * kWarps8 + (threadIdx.x >> 5); item < total;
         item += (long long)gridDim.x * kWarps8) {
        const int i = (int)(item / s.I);
        const int n = (int)(item - (long long)i * s.I);
        if (L.entry_wave[i] != wave) continue;
        const uint8_t* base = slots + (size_t)L.entry_slot[i] * s.stride;
        int4 gv[CPL], uv[CPL];
        float sg[CPL], su[CPL];
        load_row_pair_fp8<CPL>(base, s, n, lane, nchunk, false, gv, uv, sg, su);
        const uint8_t* xr = reinterpret_cast<const uint8_t*>(x + (size_t)(i / s.k) * s.H);
        const float h = row_pair_h_fp8<CPL>(gv, uv, sg, su, xr, lane, nchunk);
        if (lane == 0) hbuf[(size_t)i * s.I + n] = h;
    }
}

// Down projection of one wave (same structure as the bf16 kernel): a CTA owns
// token t and kDownRows8 rows (all in one 128-row scale block), warp w the
// entries j = w, w + 8, ...
template <int CPL>
__global__ void __launch_bounds__(kThreads8) down_fp8_kernel(LayerDev L, Shape s, const uint8_t* __restrict__ slots,
                                                            int wave, int T, const float* __restrict__ hbuf,
                                                            float* __restrict__ merged, __nv_bfloat16* __restrict__ out,
                                                            int fused) {
    __shared__ float sh_p[kMaxTopK][kDownRows8];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nchunk = s.I >> 4;
    const size_t row_bytes = (size_t)s.I;
    const int nbi = (s.I + kFp8Block - 1) / kFp8Block;
    const int blocks_per_t = (s.H + kDownRows8 - 1) / kDownRows8;
    const int t = blockIdx.x / blocks_per_t;
    const int m0 = (blockIdx.x - t * blocks_per_t) * kDownRows8;
    pdl_wait();
    pdl_trigger();
    if (t >= T) return;
    for (int j = warp; j < s.k; j += kWarps8) {
        const int i = t * s.k + j;
        if (L.entry_wave[i] != wave) {
            if (fused && lane < kDownRows8) sh_p[j][lane] = 0.f;
            continue;
        }
        const uint8_t* base = slots + (size_t)L.entry_slot[i] * s.stride;
        const float wj = L.topk_w[i];
        const uint8_t* rows = base + s.w2_off + (size_t)m0 * row_bytes;
        const float* srow = reinterpret_cast<const float*>(base + s.s2_off) + (size_t)(m0 / kFp8Block) * nbi;
        const float* h = hbuf + (size_t)i * s.I;
        int4 wv[kDownRows8][CPL];
        float sc[CPL];
#pragma unroll
        for (int r = 0; r < kDownRows8; ++r) {
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                const int idx = lane + 32 * c;
                wv[r][c] = (m0 + r < s.H && idx < nchunk) ? ldg16(rows + (size_t)r * row_bytes + 16 * (size_t)idx)
                                                          : make_int4(0, 0, 0, 0);
            }
        }
        float4 hv[CPL][4];
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            const int idx = lane + 32 * c;
            if (idx < nchunk) {
                sc[c] = __ldg(srow + (idx * 16) / kFp8Block);
#pragma unroll
                for (int v = 0; v < 4; ++v) hv[c][v] = __ldg(reinterpret_cast<const float4*>(h + 16 * idx + 4 * v));
            } else {
                sc[c] = 0.f;
#pragma unroll
                for (int v = 0; v < 4; ++v) hv[c][v] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int r = 0; r < kDownRows8; ++r) {
            float d = 0.f;
#pragma unroll
            for (int c = 0; c < CPL; ++c)
                if (lane + 32 * c < nchunk) d = fmaf(sc[c], dot16_e4m3_f32(wv[r][c], hv[c]), d);
            d = warp_sum(d);
            const float p = __fmul_rn(wj, d);
            if (lane == 0) {
                if (fused)
                    sh_p[j][r] = p;
                else if (m0 + r < s.H)
                    merged[(size_t)i * s.H + m0 + r] = p;
            }
        }
    }
    if (!fused) return;
    __syncthreads();
    if ((int)threadIdx.x < kDownRows8 && m0 + (int)threadIdx.x < s.H) {
        const int r = threadIdx.x;
        float acc = 0.f;
        for (int j = 0; j < s.k; ++j) acc = __fadd_rn(acc, sh_p[j][r]);
        out[(size_t)t * s.H + m0 + r] = __float2bfloat16_rn(acc);
    }
}

}  // namespace

cudaError_t launch_gateup_pagein_fp8(const LayerDev& L, const Shape& s, const __nv_bfloat16* x,
                                     const uint8_t* host_layer, uint8_t* slots_layer, int wave, int T, float* hbuf,
                                     int num_sms, cudaStream_t st) {
    const int grid = num_sms * 2;
    const int cpl = (s.H / 16 + 31) / 32;
    const size_t xbytes = (size_t)T * s.H * 2;
    const size_t meta = (size_t)4 * ((2 * s.K + T * s.k + 3) & ~3);
    const int stage = meta + xbytes <= (size_t)kSmemBudget8;
    const size_t smem = meta + (stage ? xbytes : 0);
#define PE_G8(C) return launch_pdl(gateup_pagein_fp8_kernel<C>, grid, kThreads8, smem, st, L, s, x, host_layer, slots_layer, wave, T, hbuf, stage)
    if (cpl <= 1) PE_G8(1);
    if (cpl <= 2) PE_G8(2);
    if (cpl <= 4) PE_G8(4);
    if (cpl <= 8) PE_G8(8);
#undef PE_G8
    return cudaErrorInvalidValue;
}

cudaError_t launch_gateup_fp8(const LayerDev& L, const Shape& s, const __nv_bfloat16* x, const uint8_t* slots_layer,
                              int wave, int T, float* hbuf, int num_sms, cudaStream_t st) {
    const long long warps = (long long)T * s.k * s.I;
    const long long blocks = (warps + kWarps8 - 1) / kWarps8;
    const int grid = (int)(blocks < (long long)num_sms * 4 ? blocks : (long long)num_sms * 4);
    if (grid <= 0) return cudaSuccess;
    const int cpl = (s.H / 16 + 31) / 32;
#define PE_U8(C) return launch_pdl(gateup_fp8_kernel<C>, grid, kThreads8, 0, st, L, s, x, slots_layer, wave, T, hbuf)
    if (cpl <= 1) PE_U8(1);
    if (cpl <= 2) PE_U8(2);
    if (cpl <= 4) PE_U8(4);
    if (cpl <= 8) PE_U8(8);
#undef PE_U8
    return cudaErrorInvalidValue;
}

cudaError_t launch_down_fp8(const LayerDev& L, const Shape& s, const uint8_t* slots_layer, int wave, int T,
                            const float* hbuf, float* merged, __nv_bfloat16* out, int fused, int num_sms,
                            cudaStream_t st) {
    (void)num_sms;
    const long long blocks = (long long)T * ((s.H + kDownRows8 - 1) / kDownRows8);
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    const int cpl = (s.I / 16 + 31) / 32;
#define PE_D8(C) return launch_pdl(down_fp8_kernel<C>, (int)blocks, kThreads8, 0, st, L, s, slots_layer, wave, T, hbuf, merged, out, fused)
    if (cpl <= 1) PE_D8(1);
    if (cpl <= 2) PE_D8(2);
    if (cpl <= 4) PE_D8(4);
#undef PE_D8
    return cudaErrorInvalidValue;
}

}  // namespace pe
