// Decode-sized expert MLP: weight-streaming GEMVs over the wave's entries.
//
// "Paged Experts" (SGLang docs), "A step: waves, page-in, merge", step 3: the
// MoE kernel runs over the wave's own entries (routed ids remapped to slots)
// without its final top-k sum, and returns every (token, expert) output
// already multiplied by its router weight.  Step 4: each entry goes into one
// merged buffer, and the merged entries get the same top-k sum.
//
// At decode sizes every expert row is read once per entry, so the kernels
// are bound by HBM bandwidth: one warp streams one weight row (16-byte loads,
// all of a lane's loads issued before any arithmetic) and reduces it with a
// fixed butterfly.  Every entry's value is computed by the same code in the
// same order wherever it lands (slot, wave, tile-mates), and the merged
// entries are fp32, so summing them in a separate kernel or inside the down
// projection gives the same bits.  That is what makes the paged output equal
// the unpaged (K = E) output bit for bit.

#include "pe_device.cuh"
#include "pe_internal.h"

namespace pe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kCopyLoads = 8;                               // 16-byte loads per lane per copy item
constexpr size_t kWarpCopy = (size_t)32 * 16 * kCopyLoads;  // 4 KiB per copy item
constexpr int kStageXBytes = 48 * 1024;                     // dynamic shared memory budget of the fused kernel

// h[i, n] = SiLU(gate_n . x_t) * (up_n . x_t) for entries i of `wave`.
// CPL = 16-byte chunks of an H-long row per lane.
template <int CPL>
__global__ void __launch_bounds__(kThreads) gateup_bf16_kernel(LayerDev L, Shape s,
                                                              const __nv_bfloat16* __restrict__ x,
                                                              const uint8_t* __restrict__ slots,
                                                              int wave, int T, float* __restrict__ hbuf) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int nchunk = s.H >> 3;
    const size_t row_bytes = (size_t)s.H * 2;
    const long long total = (long long)T * s.k * s.I;
    for (long long item = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5); item < total;
         item += (long long)gridDim.x * kWarps) {
        const int i = (int)(item / s.I);
        const int n = (int)(item - (long long)i * s.I);
        if (L.entry_wave[i] != wave) continue;
        const uint8_t* w13 = slots + (size_t)L.entry_slot[i] * s.stride + s.w13_off;
        const uint8_t* g = w13 + (size_t)n * row_bytes;
        const uint8_t* u = w13 + (size_t)(s.I + n) * row_bytes;
        const uint8_t* xr = reinterpret_cast<const uint8_t*>(x + (size_t)(i / s.k) * s.H);
        int4 gv[CPL], uv[CPL];
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            const int idx = lane + 32 * c;
            if (idx < nchunk) {
                gv[c] = ldg16(g + 16 * (size_t)idx);
                uv[c] = ldg16(u + 16 * (size_t)idx);
            } else {
                gv[c] = uv[c] = make_int4(0, 0, 0, 0);
            }
        }
        const float h = row_pair_h<CPL>(gv, uv, xr, lane, nchunk);
        if (lane == 0) hbuf[(size_t)i * s.I + n] = h;
    }
}

// Gate/up of one wave fused with its page-in (decode sizes: at most
// kFusedMaxEntries entries).  Two groups of CTAs run side by side:
//   link CTAs  - gate/up row pairs of the members paged in this wave, read
//                from the host store, written to the member's slot and used
//                for h right away; then the rest of each paged row (w2 and
//                scales) copied host -> slot in 4 KiB pieces;
//   HBM CTAs   - gate/up row pairs of the members that were already resident.
// The host link stays busy for the whole kernel while the resident experts
// stream from HBM underneath it.  For each row pair the warp computes h for
// every entry of the wave routed to that member.
//
// Dynamic shared memory: [member experts K][member slots K][entry keys nent]
// padded to a multiple of 4 ints, then, when it fits, the wave's token rows
// of x (16-byte aligned).
template <int CPL>
__global__ void __launch_bounds__(kThreads, 2) gateup_pagein_bf16_kernel(
    LayerDev L, Shape s, const __nv_bfloat16* __restrict__ x, const uint8_t* __restrict__ host,
    uint8_t* __restrict__ slots, int wave, int T, float* __restrict__ hbuf, int stage_x) {
    extern __shared__ int4 sh_dyn[];
    int32_t* sh_mexp = reinterpret_cast<int32_t*>(sh_dyn);
    int32_t* sh_mslot = sh_mexp + s.K;
    int32_t* sh_ekey = sh_mslot + s.K;  // entry's slot if it belongs to this wave, else -1
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
    if (stage_x) {  // the wave's tokens, once per CTA
        // 16-byte aligned: the metadata block is padded to a multiple of 4 ints
        int4* sx = reinterpret_cast<int4*>(sh_mexp + ((2 * s.K + nent + 3) & ~3));
        const int nvec = T * s.H / 8;
        for (int i = threadIdx.x; i < nvec; i += blockDim.x) sx[i] = ldg16(xbase + 16 * (size_t)i);
        xbase = reinterpret_cast<const uint8_t*>(sx);
    }
    __syncthreads();

    const int nchunk = s.H >> 3;
    const size_t row_bytes = (size_t)s.H * 2;
    const long long miss_rows = (long long)count * s.I;
    const size_t tail_bytes = s.copy_bytes - s.tail_off;
    const long long copies_per = (long long)((tail_bytes + kWarpCopy - 1) / kWarpCopy);
    const long long link_items = miss_rows + (long long)count * copies_per;
    const long long hbm_items = (long long)(size - count) * s.I;
    const int G = gridDim.x;
    const int Gl = link_items == 0 ? 0 : hbm_items == 0 ? G : max(1, G / 2);
    const bool link_cta = (int)blockIdx.x < Gl;
    const long long first = (long long)(link_cta ? blockIdx.x : blockIdx.x - Gl) * kWarps + warp;
    const long long stride = (long long)(link_cta ? Gl : G - Gl) * kWarps;
    const long long total = link_cta ? link_items : hbm_items;
    for (long long item = first; item < total; item += stride) {
        if (link_cta && item >= miss_rows) {
            const long long c = item - miss_rows;
            const int q = (int)(c / copies_per);
            const size_t off = s.tail_off + (size_t)(c - (long long)q * copies_per) * kWarpCopy;
            const uint8_t* src = host + (size_t)sh_mexp[q] * s.stride + off;
            uint8_t* dst = slots + (size_t)sh_mslot[q] * s.stride + off;
            const size_t nbytes = min(kWarpCopy, s.copy_bytes - off);
            int4 v[kCopyLoads];
#pragma unroll
            for (int u = 0; u < kCopyLoads; ++u) {
                const size_t o = ((size_t)u * 32 + lane) * 16;
                if (o < nbytes) v[u] = ld_nc_na(src + o);
            }
#pragma unroll
            for (int u = 0; u < kCopyLoads; ++u) {
                const size_t o = ((size_t)u * 32 + lane) * 16;
                if (o < nbytes) *reinterpret_cast<int4*>(dst + o) = v[u];
            }
            continue;
        }
        const int q = link_cta ? (int)(item / s.I) : count + (int)(item / s.I);
        const int n = (int)(item % s.I);
        const int slot = sh_mslot[q];
        uint8_t* slot_row = slots + (size_t)slot * s.stride + s.w13_off;
        const uint8_t* g = (link_cta ? host + (size_t)sh_mexp[q] * s.stride + s.w13_off : slot_row) +
                           (size_t)n * row_bytes;
        const uint8_t* u = g + (size_t)s.I * row_bytes;
        int4 gv[CPL], uv[CPL];
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            const int idx = lane + 32 * c;
            if (idx < nchunk) {
                gv[c] = link_cta ? ld_nc_na(g + 16 * (size_t)idx) : ldg16(g + 16 * (size_t)idx);
                uv[c] = link_cta ? ld_nc_na(u + 16 * (size_t)idx) : ldg16(u + 16 * (size_t)idx);
            } else {
                gv[c] = uv[c] = make_int4(0, 0, 0, 0);
            }
        }
        if (link_cta) {
            uint8_t* gd = slot_row + (size_t)n * row_bytes;
            uint8_t* ud = gd + (size_t)s.I * row_bytes;
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
                const uint8_t* xr = xbase + (size_t)(ei / s.k) * row_bytes;
                const float h = row_pair_h<CPL>(gv, uv, xr, lane, nchunk);
                if (lane == 0) hbuf[(size_t)ei * s.I + n] = h;
            }
        }
    }
}

// Down projection of one wave.  A CTA owns token t and kDownRows output
// rows; warp w handles entries j = w, w + 8, ... of t that belong to the
// wave.  The warp keeps its entry's h in registers and streams the entry's
// down rows (all kDownRows loads issued before the dot products), giving
// p_j[m] = w_tj * (down_m . h_tj) per row.  Then:
//   fused (all of t's entries are in this wave): out[t, m] = bf16(sum_j p_j[m])
//     in entry order j = 0..k-1, from shared memory;
//   else merged[t*k + j, m] = p_j[m] for the wave's entries.
// CPL = 16-byte chunks of an I-long row per lane.
constexpr int kDownRows = 8;

template <int CPL>
__global__ void __launch_bounds__(kThreads) down_bf16_kernel(LayerDev L, Shape s,
                                                            const uint8_t* __restrict__ slots, int wave,
                                                            int T, const float* __restrict__ hbuf,
                                                            float* __restrict__ merged,
                                                            __nv_bfloat16* __restrict__ out, int fused) {
    __shared__ float sh_p[kMaxTopK][kDownRows];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nchunk = s.I >> 3;
    const size_t row_bytes = (size_t)s.I * 2;
    const int blocks_per_t = (s.H + kDownRows - 1) / kDownRows;
    const int t = blockIdx.x / blocks_per_t;
    const int m0 = (blockIdx.x - t * blocks_per_t) * kDownRows;
    pdl_wait();
    pdl_trigger();
    if (t >= T) return;
    for (int j = warp; j < s.k; j += kWarps) {
        const int i = t * s.k + j;
        if (L.entry_wave[i] != wave) {
            if (fused && lane < kDownRows) sh_p[j][lane] = 0.f;  // only after a routing error
            continue;
        }
        const int slot = L.entry_slot[i];
        const float wj = L.topk_w[i];
        const uint8_t* rows = slots + (size_t)slot * s.stride + s.w2_off + (size_t)m0 * row_bytes;
        const float* h = hbuf + (size_t)i * s.I;
        int4 wv[kDownRows][CPL];
#pragma unroll
        for (int r = 0; r < kDownRows; ++r) {
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                const int idx = lane + 32 * c;
                wv[r][c] = (m0 + r < s.H && idx < nchunk) ? ldg16(rows + (size_t)r * row_bytes + 16 * (size_t)idx)
                                                          : make_int4(0, 0, 0, 0);
            }
        }
        float4 hv[CPL][2];
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            const int idx = lane + 32 * c;
            if (idx < nchunk) {
                hv[c][0] = __ldg(reinterpret_cast<const float4*>(h + 8 * idx));
                hv[c][1] = __ldg(reinterpret_cast<const float4*>(h + 8 * idx + 4));
            } else {
                hv[c][0] = hv[c][1] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int r = 0; r < kDownRows; ++r) {
            float d = 0.f;
#pragma unroll
            for (int c = 0; c < CPL; ++c)
                if (lane + 32 * c < nchunk) d = dot8_bf16_f32(wv[r][c], hv[c][0], hv[c][1], d);
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
    if ((int)threadIdx.x < kDownRows && m0 + (int)threadIdx.x < s.H) {
        const int r = threadIdx.x;
        float acc = 0.f;
        for (int j = 0; j < s.k; ++j) acc = __fadd_rn(acc, sh_p[j][r]);
        out[(size_t)t * s.H + m0 + r] = __float2bfloat16_rn(acc);
    }
}

__global__ void topk_sum_kernel(const float* __restrict__ merged, __nv_bfloat16* __restrict__ out,
                                int T, int k, int H) {
    pdl_wait();
    pdl_trigger();
    // four consecutive outputs per thread (H is a multiple of 8): 16-byte
    // loads, each output summed over j = 0..k-1 from zero as before
    const long long total4 = (long long)T * H / 4;
    for (long long q = (long long)blockIdx.x * blockDim.x + threadIdx.x; q < total4;
         q += (long long)gridDim.x * blockDim.x) {
        const int t = (int)(4 * q / H);
        const int m = (int)(4 * q - (long long)t * H);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < k; ++j) {
            const float4 v = *reinterpret_cast<const float4*>(merged + ((size_t)t * k + j) * H + m);
            acc.x = __fadd_rn(acc.x, v.x);
            acc.y = __fadd_rn(acc.y, v.y);
            acc.z = __fadd_rn(acc.z, v.z);
            acc.w = __fadd_rn(acc.w, v.w);
        }
        const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
        uint2 packed;
        packed.x = *reinterpret_cast<const uint32_t*>(&lo);
        packed.y = *reinterpret_cast<const uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(out + 4 * q) = packed;
    }
}

inline int grid_for(long long warps_needed, int num_sms) {
    const long long blocks = (warps_needed + kWarps - 1) / kWarps;
    return (int)(blocks < (long long)num_sms * 4 ? blocks : (long long)num_sms * 4);
}

}  // namespace

cudaError_t launch_gateup(const LayerDev& L, const Shape& s, const __nv_bfloat16* x,
                          const uint8_t* slots_layer, int wave, int T, float* hbuf, int num_sms,
                          cudaStream_t st) {
    const int grid = grid_for((long long)T * s.k * s.I, num_sms);
    if (grid <= 0) return cudaSuccess;
    const int cpl = (s.H / 8 + 31) / 32;
#define PE_GATEUP(C) return launch_pdl(gateup_bf16_kernel<C>, grid, kThreads, 0, st, L, s, x, slots_layer, wave, T, hbuf)
    if (cpl <= 1) PE_GATEUP(1);
    if (cpl <= 2) PE_GATEUP(2);
    if (cpl <= 4) PE_GATEUP(4);
    if (cpl <= 8) PE_GATEUP(8);
    if (cpl <= 16) PE_GATEUP(16);
#undef PE_GATEUP
    return cudaErrorInvalidValue;
}

cudaError_t launch_gateup_pagein(const LayerDev& L, const Shape& s, const __nv_bfloat16* x,
                                 const uint8_t* host_layer, uint8_t* slots_layer, int wave, int T,
                                 float* hbuf, int num_sms, cudaStream_t st) {
    const int grid = num_sms * 2;
    const int cpl = (s.H / 8 + 31) / 32;
    const size_t xbytes = (size_t)T * s.H * 2;
    const size_t meta = (size_t)4 * ((2 * s.K + T * s.k + 3) & ~3);  // same padding as the kernel
    const int stage = meta + xbytes <= (size_t)kStageXBytes;
    const size_t smem = meta + (stage ? xbytes : 0);
#define PE_GUP(C) return launch_pdl(gateup_pagein_bf16_kernel<C>, grid, kThreads, smem, st, L, s, x, host_layer, slots_layer, wave, T, hbuf, stage)
    if (cpl <= 1) PE_GUP(1);
    if (cpl <= 2) PE_GUP(2);
    if (cpl <= 4) PE_GUP(4);
    if (cpl <= 8) PE_GUP(8);
#undef PE_GUP
    return cudaErrorInvalidValue;
}

cudaError_t launch_down(const LayerDev& L, const Shape& s, const uint8_t* slots_layer, int wave,
                        int T, const float* hbuf, float* merged, __nv_bfloat16* out, int fused,
                        int num_sms, cudaStream_t st) {
    const long long blocks = (long long)T * ((s.H + kDownRows - 1) / kDownRows);
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    const int grid = (int)blocks;
    const int cpl = (s.I / 8 + 31) / 32;
#define PE_DOWN(C) return launch_pdl(down_bf16_kernel<C>, grid, kThreads, 0, st, L, s, slots_layer, wave, T, hbuf, merged, out, fused)
    if (cpl <= 1) PE_DOWN(1);
    if (cpl <= 2) PE_DOWN(2);
    if (cpl <= 3) PE_DOWN(3);
    if (cpl <= 4) PE_DOWN(4);
    if (cpl <= 8) PE_DOWN(8);
#undef PE_DOWN
    return cudaErrorInvalidValue;
}

cudaError_t launch_topk_sum(const Shape& s, const float* merged, __nv_bfloat16* out, int T,
                            cudaStream_t st) {
    const long long total = (long long)T * s.H / 4;
    const int grid = (int)((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
    if (grid <= 0) return cudaSuccess;
    return launch_pdl(topk_sum_kernel, grid, 256, 0, st, merged, out, T, s.k, s.H);
}

}  // namespace pe
