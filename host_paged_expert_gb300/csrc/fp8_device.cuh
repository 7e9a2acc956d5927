// Block-FP8 device helpers shared by the FP8 kernels: hardware E4M3 decode,
// 16-code dot products, the gate/up row pair of one expert row.
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "pe_device.cuh"
#include "pe_internal.h"

namespace pe {

__device__ __forceinline__ float2 e4m3x2(uint32_t two_codes) {
    const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two_codes & 0xffffu), __NV_E4M3);
    __half2 h;
    h = *reinterpret_cast<const __half2*>(&r);
    return __half22float2(h);
}

__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Gate and up dot products of one 16-code chunk each against the same 16
// bf16 values: pg = sum_{e<16} g_e x_e and pu likewise, each summed in
// element order from zero; the x values are widened once for both rows.
__device__ __forceinline__ void dot16x2_e4m3_bf16(int4 wg, int4 wu, int4 x0, int4 x1, float& pg, float& pu) {
    const uint32_t gv[4] = {(uint32_t)wg.x, (uint32_t)wg.y, (uint32_t)wg.z, (uint32_t)wg.w};
    const uint32_t uv[4] = {(uint32_t)wu.x, (uint32_t)wu.y, (uint32_t)wu.z, (uint32_t)wu.w};
    const uint32_t xv[8] = {(uint32_t)x0.x, (uint32_t)x0.y, (uint32_t)x0.z, (uint32_t)x0.w,
                            (uint32_t)x1.x, (uint32_t)x1.y, (uint32_t)x1.z, (uint32_t)x1.w};
    float g = 0.f, u = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float x0l = bf_lo(xv[2 * q]), x0h = bf_hi(xv[2 * q]);
        const float x1l = bf_lo(xv[2 * q + 1]), x1h = bf_hi(xv[2 * q + 1]);
        const float2 ga = e4m3x2(gv[q]), gb = e4m3x2(gv[q] >> 16);
        const float2 ua = e4m3x2(uv[q]), ub = e4m3x2(uv[q] >> 16);
        g = fmaf(ga.x, x0l, g);
        u = fmaf(ua.x, x0l, u);
        g = fmaf(ga.y, x0h, g);
        u = fmaf(ua.y, x0h, u);
        g = fmaf(gb.x, x1l, g);
        u = fmaf(ub.x, x1l, u);
        g = fmaf(gb.y, x1h, g);
        u = fmaf(ub.y, x1h, u);
    }
    pg = g;
    pu = u;
}

// sum_{e<16} w_e * h_e in element order: 16 E4M3 codes against 16 fp32 values.
__device__ __forceinline__ float dot16_e4m3_f32(int4 w, const float4 (&h)[4]) {
    const uint32_t wv[4] = {(uint32_t)w.x, (uint32_t)w.y, (uint32_t)w.z, (uint32_t)w.w};
    float p = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float2 a = e4m3x2(wv[q]), b = e4m3x2(wv[q] >> 16);
        p = fmaf(a.x, h[q].x, p);
        p = fmaf(a.y, h[q].y, p);
        p = fmaf(b.x, h[q].z, p);
        p = fmaf(b.y, h[q].w, p);
    }
    return p;
}

// h = SiLU(gate . x) * (up . x) for one FP8 gate/up row pair held by the warp
// (chunk c of lane l covers codes 16*(l + 32c) .. +15, scaled by sg[c], su[c]).
template <int CPL>
__device__ __forceinline__ float row_pair_h_fp8(const int4 (&gv)[CPL], const int4 (&uv)[CPL], const float (&sg)[CPL],
                                                const float (&su)[CPL], const uint8_t* xr, int lane, int nchunk) {
    float ag = 0.f, au = 0.f;
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
        const int idx = lane + 32 * c;
        if (idx < nchunk) {
            const int4 x0 = *reinterpret_cast<const int4*>(xr + 32 * (size_t)idx);
            const int4 x1 = *reinterpret_cast<const int4*>(xr + 32 * (size_t)idx + 16);
            float pg, pu;
            dot16x2_e4m3_bf16(gv[c], uv[c], x0, x1, pg, pu);
            ag = fmaf(sg[c], pg, ag);
            au = fmaf(su[c], pu, au);
        }
    }
    ag = warp_sum(ag);
    au = warp_sum(au);
    return __fmul_rn(silu(ag), au);
}

// Loads a gate/up row pair (codes and the lane's block scales) of expert row
// `base` (host row or slot).  stream_host selects the no-L1 load path.
template <int CPL>
__device__ __forceinline__ void load_row_pair_fp8(const uint8_t* base, const Shape& s, int n, int lane, int nchunk,
                                                  bool stream_host, int4 (&gv)[CPL], int4 (&uv)[CPL],
                                                  float (&sg)[CPL], float (&su)[CPL]) {
    const size_t H = (size_t)s.H;
    const uint8_t* g = base + s.w13_off + (size_t)n * H;
    const uint8_t* u = g + (size_t)s.I * H;
    const float* sc = reinterpret_cast<const float*>(base + s.s13_off);
    const int nbh = (s.H + kFp8Block - 1) / kFp8Block;
    const float* sgr = sc + (size_t)(n / kFp8Block) * nbh;
    const float* sur = sc + (size_t)((s.I + n) / kFp8Block) * nbh;
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
        const int idx = lane + 32 * c;
        if (idx < nchunk) {
            gv[c] = stream_host ? ld_nc_na(g + 16 * (size_t)idx) : ldg16(g + 16 * (size_t)idx);
            uv[c] = stream_host ? ld_nc_na(u + 16 * (size_t)idx) : ldg16(u + 16 * (size_t)idx);
            const int cb = (idx * 16) / kFp8Block;
            sg[c] = __ldg(sgr + cb);
            su[c] = __ldg(sur + cb);
        } else {
            gv[c] = uv[c] = make_int4(0, 0, 0, 0);
            sg[c] = su[c] = 0.f;
        }
    }
}

}  // namespace pe
