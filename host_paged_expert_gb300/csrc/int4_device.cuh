// GPTQ int4 device helpers shared by every int4 kernel: code decoding, the
// 32-code dot products, the gate/up row pair of one expert row and the down
// rows.  A weight is (q - 8) * s with q a 4-bit code and s the fp16 scale of
// its output row and group of 128 inputs.  A 16-byte chunk holds 32 codes of
// one row (input 2j in the low nibble of byte j) and never crosses a group,
// so each lane decodes its chunk, forms the chunk's dot product and adds it
// scaled by the chunk's group scale.  Every int4 GEMV kernel computes a value
// with these functions in the same order, so the GEMV paths agree bit for
// bit; the prefill converters use the pair decoding to build the bf16
// tensor-core operand.
#pragma once

#include <cuda_fp16.h>

#include "pe_device.cuh"
#include "pe_internal.h"

namespace pe {

// (q - 8) for the nibbles at bits 0 and 16 of w as a bf16 pair, exactly: the
// bf16 with bits 0x4300 | q is 128 + q, and 128 + q - 136 is representable.
__device__ __forceinline__ uint32_t i4_pair_bf16(uint32_t w) {
    const uint32_t t = (w & 0x000F000Fu) | 0x43004300u;
    const __nv_bfloat162 d = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&t), __float2bfloat162_rn(136.f));
    return *reinterpret_cast<const uint32_t*>(&d);
}

// One row's even-input and odd-input partial sums over the 8 codes of word w
// against the 8 bf16 inputs in xv[0..3] (xv[i] holds inputs 2i, 2i+1): each
// chain takes its inputs in ascending order.  The codes are decoded two at a
// time: nibbles (0,4), (1,5), (2,6), (3,7).
__device__ __forceinline__ void dot8_int4_bf16(uint32_t w, const uint32_t (&xv)[4], float& ev, float& od) {
    const uint32_t p04 = i4_pair_bf16(w), p15 = i4_pair_bf16(w >> 4);
    const uint32_t p26 = i4_pair_bf16(w >> 8), p37 = i4_pair_bf16(w >> 12);
    ev = fma_bf16_lo(p04, xv[0], ev);  // input 0
    od = fma_bf16_lh(p15, xv[0], od);  // input 1
    ev = fma_bf16_lo(p26, xv[1], ev);  // input 2
    od = fma_bf16_lh(p37, xv[1], od);  // input 3
    ev = fma_bf16_hl(p04, xv[2], ev);  // input 4
    od = fma_bf16_hh(p15, xv[2], od);  // input 5
    ev = fma_bf16_hl(p26, xv[3], ev);  // input 6
    od = fma_bf16_hh(p37, xv[3], od);  // input 7
}

// Gate and up dot products of one 32-code chunk against its 32 bf16 values
// (64 bytes at xc): pg = sum_e (g_e - 8) x_e and pu likewise.  Each is
// accumulated as an even-input and an odd-input partial sum (in input order
// within each) added at the end, so the four chains run side by side.  The
// products are exact and each step rounds once, as fmaf on the values widened
// to fp32.  The loop over the chunk's two 16-code halves stays rolled (a
// smaller body, fewer values live) and takes its words by selects: words
// indexed at run time would be placed in local memory.
__device__ __forceinline__ void dot32x2_int4_bf16(int4 wg, int4 wu, const uint8_t* xc, float& pg, float& pu) {
    float ge = 0.f, go = 0.f, ue = 0.f, uo = 0.f;
#pragma unroll 1
    for (int hf = 0; hf < 2; ++hf) {  // words 2hf and 2hf + 1: codes 16hf .. 16hf + 15
        const uint32_t g0 = hf ? (uint32_t)wg.z : (uint32_t)wg.x, g1 = hf ? (uint32_t)wg.w : (uint32_t)wg.y;
        const uint32_t u0 = hf ? (uint32_t)wu.z : (uint32_t)wu.x, u1 = hf ? (uint32_t)wu.w : (uint32_t)wu.y;
        const int4 xa = *reinterpret_cast<const int4*>(xc + 32 * hf);
        const int4 xb = *reinterpret_cast<const int4*>(xc + 32 * hf + 16);
        const uint32_t xva[4] = {(uint32_t)xa.x, (uint32_t)xa.y, (uint32_t)xa.z, (uint32_t)xa.w};
        const uint32_t xvb[4] = {(uint32_t)xb.x, (uint32_t)xb.y, (uint32_t)xb.z, (uint32_t)xb.w};
        dot8_int4_bf16(g0, xva, ge, go);
        dot8_int4_bf16(u0, xva, ue, uo);
        dot8_int4_bf16(g1, xvb, ge, go);
        dot8_int4_bf16(u1, xvb, ue, uo);
    }
    pg = __fadd_rn(ge, go);
    pu = __fadd_rn(ue, uo);
}

// (q - 8) for the nibbles at bits 0 and 16 of w as an fp16 pair, exactly: the
// fp16 with bits 0x6400 | q is 1024 + q, and 1024 + q - 1032 is representable.
__device__ __forceinline__ uint32_t i4_pair_f16(uint32_t w) {
    const uint32_t t = (w & 0x000F000Fu) | 0x64006400u;
    const __half2 d = __hsub2(*reinterpret_cast<const __half2*>(&t), __float2half2_rn(1032.f));
    return *reinterpret_cast<const uint32_t*>(&d);
}

// a * s in fp32 for the low / high fp16 half a of a pair and the fp16 scale s
// (bits in the low half of s16): the mixed-precision fma of sm_100 with a
// -0 addend, i.e. the exact product rounded once, as float(a) * float(s).
__device__ __forceinline__ float i4_lo_times(uint32_t pair, uint32_t s16) {
    float d;
    asm("{\n\t.reg .b16 al, ah, sl, sh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {sl, sh}, %2;\n\t"
        "fma.rn.f32.f16 %0, al, sl, %3;\n\t}"
        : "=f"(d)
        : "r"(pair), "r"(s16), "f"(-0.0f));
    return d;
}
__device__ __forceinline__ float i4_hi_times(uint32_t pair, uint32_t s16) {
    float d;
    asm("{\n\t.reg .b16 al, ah, sl, sh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {sl, sh}, %2;\n\t"
        "fma.rn.f32.f16 %0, ah, sl, %3;\n\t}"
        : "=f"(d)
        : "r"(pair), "r"(s16), "f"(-0.0f));
    return d;
}

// (q - 8) of the low / high code of a pair from i4_pair_bf16, as fp32.
__device__ __forceinline__ float i4_lo_f32(uint32_t pair) { return __uint_as_float(pair << 16); }
__device__ __forceinline__ float i4_hi_f32(uint32_t pair) { return __uint_as_float(pair & 0xffff0000u); }

// sum_{e<32} (q_e - 8) * h_e in input order: 32 codes against 32 fp32 values.
__device__ __forceinline__ float dot32_int4_f32(int4 w, const float4 (&h)[8]) {
    const uint32_t wv[4] = {(uint32_t)w.x, (uint32_t)w.y, (uint32_t)w.z, (uint32_t)w.w};
    float p = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t p04 = i4_pair_bf16(wv[q]), p15 = i4_pair_bf16(wv[q] >> 4);
        const uint32_t p26 = i4_pair_bf16(wv[q] >> 8), p37 = i4_pair_bf16(wv[q] >> 12);
        const float4 a = h[2 * q], b = h[2 * q + 1];
        p = fmaf(i4_lo_f32(p04), a.x, p);
        p = fmaf(i4_lo_f32(p15), a.y, p);
        p = fmaf(i4_lo_f32(p26), a.z, p);
        p = fmaf(i4_lo_f32(p37), a.w, p);
        p = fmaf(i4_hi_f32(p04), b.x, p);
        p = fmaf(i4_hi_f32(p15), b.y, p);
        p = fmaf(i4_hi_f32(p26), b.z, p);
        p = fmaf(i4_hi_f32(p37), b.w, p);
    }
    return p;
}

__device__ __forceinline__ float ld_half(const __half* p) { return __half2float(__ldg(p)); }
__device__ __forceinline__ float ldcg_half(const __half* p) {
    return __half2float(__ushort_as_half(__ldcg(reinterpret_cast<const unsigned short*>(p))));
}

// h = SiLU(gate . x) * (up . x) for one int4 gate/up row pair held by the
// warp (chunk c of lane l covers codes 32*(l + 32c) .. +31, scaled by sg[c],
// su[c]).
template <int CPL>
__device__ __forceinline__ float row_pair_h_int4(const int4 (&gv)[CPL], const int4 (&uv)[CPL], const float (&sg)[CPL],
                                                 const float (&su)[CPL], const uint8_t* xr, int lane, int nchunk) {
    float ag = 0.f, au = 0.f;
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
        const int idx = lane + 32 * c;
        if (idx < nchunk) {
            float pg, pu;
            dot32x2_int4_bf16(gv[c], uv[c], xr + 64 * (size_t)idx, pg, pu);
            ag = fmaf(sg[c], pg, ag);
            au = fmaf(su[c], pu, au);
        }
    }
    ag = warp_sum(ag);
    au = warp_sum(au);
    return __fmul_rn(silu(ag), au);
}

// Loads a gate/up row pair (codes and the lane's group scales) of expert row
// `base` (host row or slot).  stream_host selects the no-L1 load path;
// l2_only reads codes and scales past L1 (slots written in the same kernel).
template <int CPL>
__device__ __forceinline__ void load_row_pair_int4(const uint8_t* base, const Shape& s, int n, int lane, int nchunk,
                                                   bool stream_host, bool l2_only, int4 (&gv)[CPL], int4 (&uv)[CPL],
                                                   float (&sg)[CPL], float (&su)[CPL]) {
    const size_t rb = (size_t)s.H / 2;
    const uint8_t* g = base + s.w13_off + (size_t)n * rb;
    const uint8_t* u = g + (size_t)s.I * rb;
    const int ng = s.H / kInt4Group;
    const __half* sc = reinterpret_cast<const __half*>(base + s.s13_off);
    const __half* sgr = sc + (size_t)n * ng;
    const __half* sur = sc + (size_t)(s.I + n) * ng;
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
        const int idx = lane + 32 * c;
        if (idx < nchunk) {
            const int grp = (idx * 32) / kInt4Group;
            if (stream_host) {
                gv[c] = ld_nc_na(g + 16 * (size_t)idx);
                uv[c] = ld_nc_na(u + 16 * (size_t)idx);
                sg[c] = ld_half(sgr + grp);
                su[c] = ld_half(sur + grp);
            } else if (l2_only) {
                gv[c] = __ldcg(reinterpret_cast<const int4*>(g + 16 * (size_t)idx));
                uv[c] = __ldcg(reinterpret_cast<const int4*>(u + 16 * (size_t)idx));
                sg[c] = ldcg_half(sgr + grp);
                su[c] = ldcg_half(sur + grp);
            } else {
                gv[c] = ldg16(g + 16 * (size_t)idx);
                uv[c] = ldg16(u + 16 * (size_t)idx);
                sg[c] = ld_half(sgr + grp);
                su[c] = ld_half(sur + grp);
            }
        } else {
            gv[c] = uv[c] = make_int4(0, 0, 0, 0);
            sg[c] = su[c] = 0.f;
        }
    }
}

// p = w * (down_m . h) for ROWS rows m0.. of one entry, written to out_row
// (or returned in p_out when it is not null).  The down rows' codes are
// [H, I/2] bytes, their scales [H, I/128] fp16.  CPL = 16-byte chunks (32
// codes) of an I-long row per lane.  l2_only reads past L1.  HS: h is the
// entry's h staged in shared memory in the hs_pos<8> layout (else read
// through L2).
template <int CPL, int ROWS, bool HS = false, bool TR = false>
__device__ __forceinline__ void down_rows_int4(const uint8_t* w2, const __half* s2, const float* h, float wj, int m0,
                                               int H, int I, bool l2_only, float* out_row, float* p_out, int lane) {
    const int nchunk = I >> 5;
    const size_t rb = (size_t)I / 2;
    const int ng = I / kInt4Group;
    int4 wv[ROWS][CPL];
    float sc[ROWS][CPL];
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            const int idx = lane + 32 * c;
            const bool ok = m0 + r < H && idx < nchunk;
            const uint8_t* p = w2 + (size_t)(m0 + r) * rb + 16 * (size_t)idx;
            const __half* sp = s2 + (size_t)(m0 + r) * ng + (idx * 32) / kInt4Group;
            wv[r][c] = ok ? (l2_only ? __ldcg(reinterpret_cast<const int4*>(p)) : ldg16(p)) : make_int4(0, 0, 0, 0);
            sc[r][c] = ok ? (l2_only ? ldcg_half(sp) : ld_half(sp)) : 0.f;
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
            if (lane + 32 * c < nchunk) d[r] = fmaf(sc[r][c], dot32_int4_f32(wv[r][c], hv[c]), d[r]);
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
