// MXFP4 / NVFP4 device helpers shared by every FP4 kernel: E2M1 decoding,
// block-scale decoding, the 32-code dot products, the gate/up row pair of one
// expert row and the down rows.
//
// A weight is e2m1(q) * scale.  MXFP4: one E8M0 scale (2^(e - 127)) per 32
// inputs; NVFP4: one E4M3 scale per 16 inputs times the tensor's fp32 scale,
// which the expert row keeps in a 16-byte header in front of each scale grid.
// Codes are packed as for int4 (input 2j in the low nibble of byte j), so a
// 16-byte chunk holds 32 codes of one row: one MXFP4 block, two NVFP4 blocks.
// Each lane decodes its chunk, forms the dot products of the chunk's two
// 16-code halves and adds them scaled by the halves' scales (equal for
// MXFP4).  Every FP4 GEMV kernel computes a value with these functions in the
// same order, so the GEMV paths agree bit for bit; the prefill converters use
// the same decoding to build the bf16 tensor-core operand.
//
// Decoding: 2*|e2m1(q)| is an integer in {0, 1, 2, 3, 4, 6, 8, 12}; a byte
// permute looks those up for four codes at once, the bf16 with bits
// 0x4300 | n is 128 + n, and subtracting 128 leaves 2*|v| exactly; the sign
// bit is copied in.  The factor 1/2 is folded into the scales (exactly).
#pragma once

#include <cuda_fp16.h>

#include "fp8_device.cuh"
#include "int4_device.cuh"
#include "pe_device.cuh"
#include "pe_internal.h"

namespace pe {

// Bytes in front of a scale grid: the NVFP4 tensor scale (fp32, then padding).
__host__ __device__ constexpr int fp4_scale_header(int fmt) { return fmt == PE_NVFP4 ? 16 : 0; }
// Inputs per block scale, and scale bytes per 32-code chunk.
__host__ __device__ constexpr int fp4_block(int fmt) { return fmt == PE_NVFP4 ? kNvfp4Block : kMxfp4Block; }

// Four bf16 pairs holding 2*e2m1 of the eight codes of w (code j in nibble j):
// p[i] = (code 2i in the low half, code 2i+1 in the high half), exactly.
__device__ __forceinline__ void e2m1x8_bf16x2(uint32_t w, uint32_t (&p)[4]) {
    const uint32_t mag = w & 0x77777777u;
    // bytes 0..7 of the table: 2*|v| of magnitudes 0..7
    const uint32_t lo = __byte_perm(0x03020100u, 0x0C080604u, mag);        // codes 0..3, one byte each
    const uint32_t hi = __byte_perm(0x03020100u, 0x0C080604u, mag >> 16);  // codes 4..7
    const __nv_bfloat162 k128 = __float2bfloat162_rn(128.f);
    const uint32_t q[4] = {__byte_perm(lo, 0x43u, 0x4140u), __byte_perm(lo, 0x43u, 0x4342u),
                           __byte_perm(hi, 0x43u, 0x4140u), __byte_perm(hi, 0x43u, 0x4342u)};
    // sign of code 2i (bit 8i+3 of w) to bit 15, of code 2i+1 (bit 8i+7) to bit 31
    const uint32_t sg[4] = {((w << 12) & 0x8000u) | ((w << 24) & 0x80000000u),
                            ((w << 4) & 0x8000u) | ((w << 16) & 0x80000000u),
                            ((w >> 4) & 0x8000u) | ((w << 8) & 0x80000000u),
                            ((w >> 12) & 0x8000u) | (w & 0x80000000u)};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 d = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&q[i]), k128);
        p[i] = *reinterpret_cast<const uint32_t*>(&d) | sg[i];
    }
}

// Half of an E8M0 scale, 2^(e - 128), as fp32 (fp32 subnormals for e < 2;
// NaN for e = 255).
__device__ __forceinline__ float e8m0_half(uint32_t e) {
    e &= 0xFFu;
    if (e == 255u) return __uint_as_float(0x7FC00000u);
    return e >= 2u ? __uint_as_float((e - 1u) << 23) : __uint_as_float(0x00200000u << e);
}

// The two block scales (times 1/2) of a 32-code chunk: codes 0..15 in .x,
// 16..31 in .y.  grid: the scale grid of the code's row; idx: chunk index in
// the row; g_half: NVFP4 tensor scale times 1/2 (unused for MXFP4).
template <int FMT>
__device__ __forceinline__ float2 fp4_chunk_scales(const uint8_t* grid_row, int idx, float g_half, bool l2_only) {
    if constexpr (FMT == PE_NVFP4) {
        const unsigned short* p = reinterpret_cast<const unsigned short*>(grid_row) + idx;
        const uint32_t two = l2_only ? __ldcg(p) : __ldg(p);
        const float2 v = e4m3x2(two);
        return make_float2(v.x * g_half, v.y * g_half);
    } else {
        const uint32_t e = l2_only ? __ldcg(grid_row + idx) : __ldg(grid_row + idx);
        const float s = e8m0_half(e);
        return make_float2(s, s);
    }
}

// NVFP4 tensor scale times 1/2 from a scale header (1 for MXFP4).
template <int FMT>
__device__ __forceinline__ float fp4_global_half(const uint8_t* scale_region, bool l2_only) {
    if constexpr (FMT == PE_NVFP4) {
        const float* g = reinterpret_cast<const float*>(scale_region);
        return 0.5f * (l2_only ? __ldcg(g) : __ldg(g));
    } else {
        return 1.f;
    }
}

// Gate and up dot products of one 32-code chunk against its 32 bf16 values
// (64 bytes at xc), each as the sums over codes 0..15 and 16..31 (2*v units):
// every half as an even-input and an odd-input chain in input order, added at
// the end.  Products are exact and each step rounds once.  The loop over the
// halves stays rolled (fewer decoded pairs live) and takes its words by
// selects: words indexed at run time would be placed in local memory.
__device__ __forceinline__ void dot32x2_fp4_bf16(int4 wg, int4 wu, const uint8_t* xc, float2& pg, float2& pu) {
    float g0 = 0.f, g1 = 0.f, u0 = 0.f, u1 = 0.f;
#pragma unroll 1
    for (int hf = 0; hf < 2; ++hf) {  // words 2hf and 2hf + 1 against x at xc + 32hf
        float ge = 0.f, go = 0.f, ue = 0.f, uo = 0.f;
        const uint32_t gw[2] = {hf ? (uint32_t)wg.z : (uint32_t)wg.x, hf ? (uint32_t)wg.w : (uint32_t)wg.y};
        const uint32_t uw[2] = {hf ? (uint32_t)wu.z : (uint32_t)wu.x, hf ? (uint32_t)wu.w : (uint32_t)wu.y};
#pragma unroll
        for (int q = 0; q < 2; ++q) {  // word 2hf + q: codes 8(2hf + q) .. +7
            const int4 xq = *reinterpret_cast<const int4*>(xc + 32 * hf + 16 * q);
            const uint32_t xv[4] = {(uint32_t)xq.x, (uint32_t)xq.y, (uint32_t)xq.z, (uint32_t)xq.w};
            uint32_t pgv[4], puv[4];
            e2m1x8_bf16x2(gw[q], pgv);
            e2m1x8_bf16x2(uw[q], puv);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                ge = fma_bf16_lo(pgv[i], xv[i], ge);
                go = fma_bf16_hh(pgv[i], xv[i], go);
                ue = fma_bf16_lo(puv[i], xv[i], ue);
                uo = fma_bf16_hh(puv[i], xv[i], uo);
            }
        }
        const float gs = __fadd_rn(ge, go), us = __fadd_rn(ue, uo);
        if (hf) {
            g1 = gs;
            u1 = us;
        } else {
            g0 = gs;
            u0 = us;
        }
    }
    pg = make_float2(g0, g1);
    pu = make_float2(u0, u1);
}

// The two 16-code halves of sum_{e<32} 2*v_e * h_e (input order within each):
// 32 codes against 32 fp32 values.
__device__ __forceinline__ float2 dot32_fp4_f32(int4 w, const float4 (&h)[8]) {
    const uint32_t wv[4] = {(uint32_t)w.x, (uint32_t)w.y, (uint32_t)w.z, (uint32_t)w.w};
    float d[2] = {0.f, 0.f};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t p[4];
        e2m1x8_bf16x2(wv[q], p);
        const float4 a = h[2 * q], b = h[2 * q + 1];  // inputs 8q..8q+3, 8q+4..8q+7
        float& acc = d[q >> 1];
        acc = fmaf(bf_lo(p[0]), a.x, acc);
        acc = fmaf(bf_hi(p[0]), a.y, acc);
        acc = fmaf(bf_lo(p[1]), a.z, acc);
        acc = fmaf(bf_hi(p[1]), a.w, acc);
        acc = fmaf(bf_lo(p[2]), b.x, acc);
        acc = fmaf(bf_hi(p[2]), b.y, acc);
        acc = fmaf(bf_lo(p[3]), b.z, acc);
        acc = fmaf(bf_hi(p[3]), b.w, acc);
    }
    return make_float2(d[0], d[1]);
}

// h = SiLU(gate . x) * (up . x) for one FP4 gate/up row pair held by the
// warp (chunk c of lane l covers codes 32*(l + 32c) .. +31 with the block
// scales sg[c], su[c], each times 1/2).
template <int CPL>
__device__ __forceinline__ float row_pair_h_fp4(const int4 (&gv)[CPL], const int4 (&uv)[CPL], const float2 (&sg)[CPL],
                                                const float2 (&su)[CPL], const uint8_t* xr, int lane, int nchunk) {
    float ag = 0.f, au = 0.f;
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
        const int idx = lane + 32 * c;
        if (idx < nchunk) {
            float2 pg, pu;
            dot32x2_fp4_bf16(gv[c], uv[c], xr + 64 * (size_t)idx, pg, pu);
            ag = fmaf(sg[c].y, pg.y, fmaf(sg[c].x, pg.x, ag));
            au = fmaf(su[c].y, pu.y, fmaf(su[c].x, pu.x, au));
        }
    }
    ag = warp_sum(ag);
    au = warp_sum(au);
    return __fmul_rn(silu(ag), au);
}

// Loads a gate/up row pair (codes and the lane's chunk scales) of expert row
// `base` (host row or slot).  stream_host selects the no-L1 load path;
// l2_only reads codes and scales past L1 (slots written in the same kernel).
template <int FMT, int CPL>
__device__ __forceinline__ void load_row_pair_fp4(const uint8_t* base, const Shape& s, int n, int lane, int nchunk,
                                                  bool stream_host, bool l2_only, int4 (&gv)[CPL], int4 (&uv)[CPL],
                                                  float2 (&sg)[CPL], float2 (&su)[CPL]) {
    const size_t rb = (size_t)s.H / 2;
    const uint8_t* g = base + s.w13_off + (size_t)n * rb;
    const uint8_t* u = g + (size_t)s.I * rb;
    const size_t srow = (size_t)s.H / fp4_block(FMT);  // scale bytes per row
    const uint8_t* region = base + s.s13_off;
    const uint8_t* grid = region + fp4_scale_header(FMT);
    const bool l2 = l2_only && !stream_host;
    const float gh = fp4_global_half<FMT>(region, l2);
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
        const int idx = lane + 32 * c;
        if (idx < nchunk) {
            if (stream_host) {
                gv[c] = ld_nc_na(g + 16 * (size_t)idx);
                uv[c] = ld_nc_na(u + 16 * (size_t)idx);
            } else if (l2_only) {
                gv[c] = __ldcg(reinterpret_cast<const int4*>(g + 16 * (size_t)idx));
                uv[c] = __ldcg(reinterpret_cast<const int4*>(u + 16 * (size_t)idx));
            } else {
                gv[c] = ldg16(g + 16 * (size_t)idx);
                uv[c] = ldg16(u + 16 * (size_t)idx);
            }
            sg[c] = fp4_chunk_scales<FMT>(grid + (size_t)n * srow, idx, gh, l2);
            su[c] = fp4_chunk_scales<FMT>(grid + (size_t)(s.I + n) * srow, idx, gh, l2);
        } else {
            gv[c] = uv[c] = make_int4(0, 0, 0, 0);
            sg[c] = su[c] = make_float2(0.f, 0.f);
        }
    }
}

// p = w * (down_m . h) for ROWS rows m0.. of one entry, written to out_row
// (or returned in p_out when it is not null).  The down rows' codes are
// [H, I/2] bytes, their scale grid [H, I/block] after the header.  CPL =
// 16-byte chunks (32 codes) of an I-long row per lane.  l2_only reads past L1.
// HS: h staged in shared memory in the hs_pos<8> layout (else read through L2).
template <int FMT, int CPL, int ROWS, bool HS = false, bool TR = false>
__device__ __forceinline__ void down_rows_fp4(const uint8_t* w2, const uint8_t* s2_region, const float* h, float wj,
                                              int m0, int H, int I, bool l2_only, float* out_row, float* p_out,
                                              int lane) {
    const int nchunk = I >> 5;
    const size_t rb = (size_t)I / 2;
    const size_t srow = (size_t)I / fp4_block(FMT);
    const uint8_t* grid = s2_region + fp4_scale_header(FMT);
    const float gh = fp4_global_half<FMT>(s2_region, l2_only);
    int4 wv[ROWS][CPL];
    float2 sc[ROWS][CPL];
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            const int idx = lane + 32 * c;
            const bool ok = m0 + r < H && idx < nchunk;
            const uint8_t* p = w2 + (size_t)(m0 + r) * rb + 16 * (size_t)idx;
            wv[r][c] = ok ? (l2_only ? __ldcg(reinterpret_cast<const int4*>(p)) : ldg16(p)) : make_int4(0, 0, 0, 0);
            sc[r][c] = ok ? fp4_chunk_scales<FMT>(grid + (size_t)(m0 + r) * srow, idx, gh, l2_only)
                          : make_float2(0.f, 0.f);
        }
    float4 hv[CPL][8];
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
        const int idx = lane + 32 * c;
#pragma unroll
        for (int v = 0; v < 8; ++v)
            hv[c][v] = idx >= nchunk ? make_float4(0.f, 0.f, 0.f, 0.f)
                       : HS ? reinterpret_cast<const float4*>(h)[hs_pos<8>(idx, v)]
                            : __ldcg(reinterpret_cast<const float4*>(h + 32 * idx + 4 * v));
    }
    float d[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        d[r] = 0.f;
#pragma unroll
        for (int c = 0; c < CPL; ++c)
            if (lane + 32 * c < nchunk) {
                const float2 hh = dot32_fp4_f32(wv[r][c], hv[c]);
                d[r] = fmaf(sc[r][c].y, hh.y, fmaf(sc[r][c].x, hh.x, d[r]));
            }
    }
    if constexpr (TR) {  // row totals by the transposed butterfly, written by one lane each
        constexpr int SH = ROWS == 8 ? 2 : ROWS == 4 ? 3 : ROWS == 2 ? 4 : 5;
        const float t = warp_sum_rows<ROWS>(d, lane);
        const int r = lane >> SH;
        if ((lane & ((1 << SH) - 1)) == 0 && m0 + r < H) out_row[m0 + r] = __fmul_rn(wj, t);
    } else {
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            const float p = __fmul_rn(wj, warp_sum(d[r]));
            if (p_out) p_out[r] = p;
            if (lane == 0 && out_row && m0 + r < H) out_row[m0 + r] = p;
        }
    }
}

}  // namespace pe

namespace pe {

// The per-format operations of the 4-bit GEMV kernels (GPTQ int4, MXFP4,
// NVFP4): their code layout is shared, the decoding and scales differ.
template <int FMT>
struct Q4Ops;

template <>
struct Q4Ops<PE_INT4_GPTQ> {
    using Scale = float;
    template <int CPL>
    static __device__ __forceinline__ void load(const uint8_t* base, const Shape& s, int n, int lane, int nchunk,
                                                bool stream_host, bool l2_only, int4 (&gv)[CPL], int4 (&uv)[CPL],
                                                Scale (&sg)[CPL], Scale (&su)[CPL]) {
        load_row_pair_int4<CPL>(base, s, n, lane, nchunk, stream_host, l2_only, gv, uv, sg, su);
    }
    template <int CPL>
    static __device__ __forceinline__ float h(const int4 (&gv)[CPL], const int4 (&uv)[CPL], const Scale (&sg)[CPL],
                                              const Scale (&su)[CPL], const uint8_t* xr, int lane, int nchunk) {
        return row_pair_h_int4<CPL>(gv, uv, sg, su, xr, lane, nchunk);
    }
    template <int CPL, int ROWS>
    static __device__ __forceinline__ void down(const uint8_t* base, const Shape& s, const float* h, float wj, int m0,
                                                bool l2_only, float* out_row, float* p_out, int lane) {
        down_rows_int4<CPL, ROWS>(base + s.w2_off, reinterpret_cast<const __half*>(base + s.s2_off), h, wj, m0, s.H,
                                  s.I, l2_only, out_row, p_out, lane);
    }
};

template <int FMT>
struct Q4OpsFp4 {
    using Scale = float2;
    template <int CPL>
    static __device__ __forceinline__ void load(const uint8_t* base, const Shape& s, int n, int lane, int nchunk,
                                                bool stream_host, bool l2_only, int4 (&gv)[CPL], int4 (&uv)[CPL],
                                                Scale (&sg)[CPL], Scale (&su)[CPL]) {
        load_row_pair_fp4<FMT, CPL>(base, s, n, lane, nchunk, stream_host, l2_only, gv, uv, sg, su);
    }
    template <int CPL>
    static __device__ __forceinline__ float h(const int4 (&gv)[CPL], const int4 (&uv)[CPL], const Scale (&sg)[CPL],
                                              const Scale (&su)[CPL], const uint8_t* xr, int lane, int nchunk) {
        return row_pair_h_fp4<CPL>(gv, uv, sg, su, xr, lane, nchunk);
    }
    template <int CPL, int ROWS>
    static __device__ __forceinline__ void down(const uint8_t* base, const Shape& s, const float* h, float wj, int m0,
                                                bool l2_only, float* out_row, float* p_out, int lane) {
        down_rows_fp4<FMT, CPL, ROWS>(base + s.w2_off, base + s.s2_off, h, wj, m0, s.H, s.I, l2_only, out_row, p_out,
                                      lane);
    }
};

template <>
struct Q4Ops<PE_MXFP4> : Q4OpsFp4<PE_MXFP4> {};
template <>
struct Q4Ops<PE_NVFP4> : Q4OpsFp4<PE_NVFP4> {};

}  // namespace pe
