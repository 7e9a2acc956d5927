// 4-bit expert MLP for decode sizes: GPTQ int4 ("Paged Experts", SGLang docs,
// "Supported Configurations and Limitations") and MXFP4 / NVFP4 ("SGLang
// Paged Experts: corré MoE más grandes que tu VRAM", "¿Qué es la paginación
// de expertos…?").  GPTQ int4: W[n, k] = (q[n, k] - 8) * s[n][k / 128] with
// fp16 scales; MXFP4: W = e2m1(q) * 2^(e - 127) per 32 inputs; NVFP4:
// W = e2m1(q) * e4m3(s) * g per 16 inputs.  Activations stay bf16 and
// accumulation is fp32.
//
// The kernels mirror the block-FP8 ones: gate/up with the page-in fused in,
// the same on resident slots only, and the down projection with the top-k
// sum.  All arithmetic is in int4_device.cuh and fp4_device.cuh (Q4Ops),
// shared with the one-kernel decode step.  Scales are read from the same
// place as the codes (host row for a page-in, slot for a hit), so a slot
// never pairs one expert's codes with another's scales.

#include <cuda_fp16.h>

#include "fp4_device.cuh"
#include "int4_device.cuh"
#include "pe_device.cuh"
#include "pe_internal.h"

namespace pe {
namespace {

constexpr int kThreads4 = 256;
constexpr int kWarps4 = kThreads4 / 32;
constexpr int kCopyLoads4 = 8;
constexpr size_t kWarpCopy4 = (size_t)32 * 16 * kCopyLoads4;
constexpr int kDownRows4 = 8;
// rows of a down item: FP4's two scales per chunk take registers int4 does not need
template <int FMT>
constexpr int down_rows4() { return FMT == PE_INT4_GPTQ ? kDownRows4 : 4; }
constexpr int kSmemBudget4 = 48 * 1024;

// Gate/up of one wave fused with its page-in; same work split as the bf16
// kernel (link CTAs: page-in rows used for h, then the rest of each paged row;
// HBM CTAs: resident members' rows).
template <int FMT, int CPL>
__global__ void __launch_bounds__(kThreads4, 2) gateup_pagein_q4_kernel(
    LayerDev L, Shape s, const __nv_bfloat16* __restrict__ x, const uint8_t* __restrict__ host,
    uint8_t* __restrict__ slots, int wave, int T, float* __restrict__ hbuf, int stage_x) {
    extern __shared__ int4 sh_dyn4[];
    int32_t* sh_mexp = reinterpret_cast<int32_t*>(sh_dyn4);
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

    const int nchunk = s.H >> 5;
    const size_t xrow = (size_t)s.H * 2;
    const long long miss_rows = (long long)count * s.I;
    const size_t tail_bytes = s.copy_bytes - s.tail_off;
    const long long copies_per = (long long)((tail_bytes + kWarpCopy4 - 1) / kWarpCopy4);
    const long long link_items = miss_rows + (long long)count * copies_per;
    const long long hbm_items = (long long)(size - count) * s.I;
    const int G = gridDim.x;
    const int Gl = link_items == 0 ? 0 : hbm_items == 0 ? G : max(1, G / 2);
    const bool link_cta = (int)blockIdx.x < Gl;
    const long long first = (long long)(link_cta ? blockIdx.x : blockIdx.x - Gl) * kWarps4 + warp;
    const long long stride = (long long)(link_cta ? Gl : G - Gl) * kWarps4;
    const long long total = link_cta ? link_items : hbm_items;
    for (long long item = first; item < total; item += stride) {
        if (link_cta && item >= miss_rows) {
            const long long c = item - miss_rows;
            const int q = (int)(c / copies_per);
            const size_t off = s.tail_off + (size_t)(c - (long long)q * copies_per) * kWarpCopy4;
            const uint8_t* src = host + (size_t)sh_mexp[q] * s.stride + off;
            uint8_t* dst = slots + (size_t)sh_mslot[q] * s.stride + off;
            const size_t nbytes = min(kWarpCopy4, s.copy_bytes - off);
            int4 v[kCopyLoads4];
#pragma unroll
            for (int u = 0; u < kCopyLoads4; ++u) {
                const size_t o = ((size_t)u * 32 + lane) * 16;
                if (o < nbytes) v[u] = ld_nc_na(src + o);
            }
#pragma unroll
            for (int u = 0; u < kCopyLoads4; ++u) {
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
        typename Q4Ops<FMT>::Scale sg[CPL], su[CPL];
        Q4Ops<FMT>::template load<CPL>(base, s, n, lane, nchunk, link_cta, false, gv, uv, sg, su);
        if (link_cta) {
            uint8_t* gd = slot_base + s.w13_off + (size_t)n * (s.H / 2);
            uint8_t* ud = gd + (size_t)s.I * (s.H / 2);
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
                const float h =
                    Q4Ops<FMT>::template h<CPL>(gv, uv, sg, su, xbase + (size_t)(ei / s.k) * xrow, lane, nchunk);
                if (lane == 0) hbuf[(size_t)ei * s.I + n] = h;
            }
        }
    }
}

// Gate/up of one wave from the slots only (after a separate page-in): one
// warp per (entry, row).
template <int FMT, int CPL>
__global__ void __launch_bounds__(kThreads4) gateup_q4_kernel(LayerDev L, Shape s, const __nv_bfloat16* __restrict__ x,
                                                              const uint8_t* __restrict__ slots, int wave, int T,
                                                              float* __restrict__ hbuf) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int nchunk = s.H >> 5;
    const long long total = (long long)T * s.k * s.I;
    for (long long item = (long long)blockIdx.x * kWarps4 + (threadIdx.x >> 5); item < total;
         item += (long long)gridDim.x * kWarps4) {
        const int i = (int)(item / s.I);
        const int n = (int)(item - (long long)i * s.I);
        if (L.entry_wave[i] != wave) continue;
        const uint8_t* base = slots + (size_t)L.entry_slot[i] * s.stride;
        int4 gv[CPL], uv[CPL];
        typename Q4Ops<FMT>::Scale sg[CPL], su[CPL];
        Q4Ops<FMT>::template load<CPL>(base, s, n, lane, nchunk, false, false, gv, uv, sg, su);
        const uint8_t* xr = reinterpret_cast<const uint8_t*>(x + (size_t)(i / s.k) * s.H);
        const float h = Q4Ops<FMT>::template h<CPL>(gv, uv, sg, su, xr, lane, nchunk);
        if (lane == 0) hbuf[(size_t)i * s.I + n] = h;
    }
}

// Down projection of one wave (same structure as the bf16 kernel): a CTA owns
// token t and kDownRows4 rows, warp w the entries j = w, w + 8, ...
template <int FMT, int CPL, int ROWS = down_rows4<FMT>()>
__global__ void __launch_bounds__(kThreads4) down_q4_kernel(LayerDev L, Shape s, const uint8_t* __restrict__ slots,
                                                             int wave, int T, const float* __restrict__ hbuf,
                                                             float* __restrict__ merged, __nv_bfloat16* __restrict__ out,
                                                             int fused) {
    __shared__ float sh_p[kMaxTopK][ROWS];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int blocks_per_t = (s.H + ROWS - 1) / ROWS;
    const int t = blockIdx.x / blocks_per_t;
    const int m0 = (blockIdx.x - t * blocks_per_t) * ROWS;
    pdl_wait();
    pdl_trigger();
    if (t >= T) return;
    for (int j = warp; j < s.k; j += kWarps4) {
        const int i = t * s.k + j;
        if (L.entry_wave[i] != wave) {
            if (fused && lane < ROWS) sh_p[j][lane] = 0.f;
            continue;
        }
        const uint8_t* base = slots + (size_t)L.entry_slot[i] * s.stride;
        float p[ROWS];
        Q4Ops<FMT>::template down<CPL, ROWS>(base, s, hbuf + (size_t)i * s.I, L.topk_w[i], m0, false,
                                                   fused ? nullptr : merged + (size_t)i * s.H, p, lane);
        if (fused && lane == 0) {
#pragma unroll
            for (int r = 0; r < ROWS; ++r) sh_p[j][r] = p[r];
        }
    }
    if (!fused) return;
    __syncthreads();
    if ((int)threadIdx.x < ROWS && m0 + (int)threadIdx.x < s.H) {
        const int r = threadIdx.x;
        float acc = 0.f;
        for (int j = 0; j < s.k; ++j) acc = __fadd_rn(acc, sh_p[j][r]);
        out[(size_t)t * s.H + m0 + r] = __float2bfloat16_rn(acc);
    }
}


template <int FMT>
cudaError_t gateup_pagein_q4(const LayerDev& L, const Shape& s, const __nv_bfloat16* x, const uint8_t* host_layer,
                             uint8_t* slots_layer, int wave, int T, float* hbuf, int num_sms, cudaStream_t st) {
    const int grid = num_sms * 2;
    const int cpl = (s.H / 32 + 31) / 32;
    const size_t xbytes = (size_t)T * s.H * 2;
    const size_t meta = (size_t)4 * ((2 * s.K + T * s.k + 3) & ~3);
    const int stage = meta + xbytes <= (size_t)kSmemBudget4;
    const size_t smem = meta + (stage ? xbytes : 0);
#define PE_G4(C) return launch_pdl(gateup_pagein_q4_kernel<FMT, C>, grid, kThreads4, smem, st, L, s, x, host_layer, slots_layer, wave, T, hbuf, stage)
    if (cpl <= 1) PE_G4(1);
    if (cpl <= 2) PE_G4(2);
    if (cpl <= 4) PE_G4(4);
    if (cpl <= 8) PE_G4(8);
#undef PE_G4
    return cudaErrorInvalidValue;
}

template <int FMT>
cudaError_t gateup_q4(const LayerDev& L, const Shape& s, const __nv_bfloat16* x, const uint8_t* slots_layer, int wave,
                      int T, float* hbuf, int num_sms, cudaStream_t st) {
    const long long warps = (long long)T * s.k * s.I;
    const long long blocks = (warps + kWarps4 - 1) / kWarps4;
    const int grid = (int)(blocks < (long long)num_sms * 4 ? blocks : (long long)num_sms * 4);
    if (grid <= 0) return cudaSuccess;
    const int cpl = (s.H / 32 + 31) / 32;
#define PE_U4(C) return launch_pdl(gateup_q4_kernel<FMT, C>, grid, kThreads4, 0, st, L, s, x, slots_layer, wave, T, hbuf)
    if (cpl <= 1) PE_U4(1);
    if (cpl <= 2) PE_U4(2);
    if (cpl <= 4) PE_U4(4);
    if (cpl <= 8) PE_U4(8);
#undef PE_U4
    return cudaErrorInvalidValue;
}

template <int FMT>
cudaError_t down_q4(const LayerDev& L, const Shape& s, const uint8_t* slots_layer, int wave, int T, const float* hbuf,
                    float* merged, __nv_bfloat16* out, int fused, cudaStream_t st) {
    const long long blocks = (long long)T * ((s.H + down_rows4<FMT>() - 1) / down_rows4<FMT>());
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    const int cpl = (s.I / 32 + 31) / 32;
#define PE_D4(C) return launch_pdl(down_q4_kernel<FMT, C>, (int)blocks, kThreads4, 0, st, L, s, slots_layer, wave, T, hbuf, merged, out, fused)
    if (cpl <= 1) PE_D4(1);
    if (cpl <= 2) PE_D4(2);
    if (cpl <= 4) PE_D4(4);
#undef PE_D4
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_gateup_pagein_q4(const LayerDev& L, const Shape& s, const __nv_bfloat16* x,
                                    const uint8_t* host_layer, uint8_t* slots_layer, int wave, int T, float* hbuf,
                                    int num_sms, cudaStream_t st) {
    if (s.dtype == PE_MXFP4) return gateup_pagein_q4<PE_MXFP4>(L, s, x, host_layer, slots_layer, wave, T, hbuf, num_sms, st);
    if (s.dtype == PE_NVFP4) return gateup_pagein_q4<PE_NVFP4>(L, s, x, host_layer, slots_layer, wave, T, hbuf, num_sms, st);
    return gateup_pagein_q4<PE_INT4_GPTQ>(L, s, x, host_layer, slots_layer, wave, T, hbuf, num_sms, st);
}

cudaError_t launch_gateup_q4(const LayerDev& L, const Shape& s, const __nv_bfloat16* x, const uint8_t* slots_layer,
                             int wave, int T, float* hbuf, int num_sms, cudaStream_t st) {
    if (s.dtype == PE_MXFP4) return gateup_q4<PE_MXFP4>(L, s, x, slots_layer, wave, T, hbuf, num_sms, st);
    if (s.dtype == PE_NVFP4) return gateup_q4<PE_NVFP4>(L, s, x, slots_layer, wave, T, hbuf, num_sms, st);
    return gateup_q4<PE_INT4_GPTQ>(L, s, x, slots_layer, wave, T, hbuf, num_sms, st);
}

cudaError_t launch_down_q4(const LayerDev& L, const Shape& s, const uint8_t* slots_layer, int wave, int T,
                           const float* hbuf, float* merged, __nv_bfloat16* out, int fused, int num_sms,
                           cudaStream_t st) {
    (void)num_sms;
    if (s.dtype == PE_MXFP4) return down_q4<PE_MXFP4>(L, s, slots_layer, wave, T, hbuf, merged, out, fused, st);
    if (s.dtype == PE_NVFP4) return down_q4<PE_NVFP4>(L, s, slots_layer, wave, T, hbuf, merged, out, fused, st);
    return down_q4<PE_INT4_GPTQ>(L, s, slots_layer, wave, T, hbuf, merged, out, fused, st);
}

}  // namespace pe
