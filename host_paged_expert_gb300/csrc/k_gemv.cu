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

#include "pe_internal.h"

namespace pe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ int4 ldg16(const void* p) { return __ldg(reinterpret_cast<const int4*>(p)); }

// acc += sum of the 8 bf16 products of w and x, in element order.
__device__ __forceinline__ float dot8_bf16(int4 w, int4 x, float acc) {
    const uint32_t wv[4] = {(uint32_t)w.x, (uint32_t)w.y, (uint32_t)w.z, (uint32_t)w.w};
    const uint32_t xv[4] = {(uint32_t)x.x, (uint32_t)x.y, (uint32_t)x.z, (uint32_t)x.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        acc = fmaf(__uint_as_float(wv[q] << 16), __uint_as_float(xv[q] << 16), acc);
        acc = fmaf(__uint_as_float(wv[q] & 0xffff0000u), __uint_as_float(xv[q] & 0xffff0000u), acc);
    }
    return acc;
}

// acc += sum of the 8 products of bf16 weights and fp32 activations h[0..7].
__device__ __forceinline__ float dot8_bf16_f32(int4 w, float4 h0, float4 h1, float acc) {
    const uint32_t wv[4] = {(uint32_t)w.x, (uint32_t)w.y, (uint32_t)w.z, (uint32_t)w.w};
    const float hv[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        acc = fmaf(__uint_as_float(wv[q] << 16), hv[2 * q], acc);
        acc = fmaf(__uint_as_float(wv[q] & 0xffff0000u), hv[2 * q + 1], acc);
    }
    return acc;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float silu(float g) { return __fdiv_rn(g, __fadd_rn(1.f, expf(-g))); }

// h[i, n] = SiLU(gate_n . x_t) * (up_n . x_t) for entries i of `wave`.
// CPL = 16-byte chunks of an H-long row per lane.
template <int CPL>
__global__ void __launch_bounds__(kThreads) gateup_bf16_kernel(LayerDev L, Shape s,
                                                              const __nv_bfloat16* __restrict__ x,
                                                              const uint8_t* __restrict__ slots,
                                                              int wave, int T, float* __restrict__ hbuf) {
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
        int4 gv[CPL], uv[CPL], xv[CPL];
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            const int idx = lane + 32 * c;
            if (idx < nchunk) {
                gv[c] = ldg16(g + 16 * (size_t)idx);
                uv[c] = ldg16(u + 16 * (size_t)idx);
                xv[c] = ldg16(xr + 16 * (size_t)idx);
            } else {
                gv[c] = uv[c] = xv[c] = make_int4(0, 0, 0, 0);
            }
        }
        float ag = 0.f, au = 0.f;
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            ag = dot8_bf16(gv[c], xv[c], ag);
            au = dot8_bf16(uv[c], xv[c], au);
        }
        ag = warp_sum(ag);
        au = warp_sum(au);
        if (lane == 0) hbuf[(size_t)i * s.I + n] = __fmul_rn(silu(ag), au);
    }
}

// One warp per (token t, output row m).  For each entry j of t in `wave`:
// p_j = w_tj * (down_m . h_tj).  fused: out[t, m] = bf16(sum_j p_j) (all
// entries in this wave); else merged[t*k + j, m] = p_j.
// CPL = 16-byte chunks of an I-long row per lane; entries go 8 at a time.
template <int CPL>
__global__ void __launch_bounds__(kThreads) down_bf16_kernel(LayerDev L, Shape s,
                                                            const uint8_t* __restrict__ slots, int wave,
                                                            int T, const float* __restrict__ hbuf,
                                                            float* __restrict__ merged,
                                                            __nv_bfloat16* __restrict__ out, int fused) {
    constexpr int JB = 8;
    const int lane = threadIdx.x & 31;
    const int nchunk = s.I >> 3;
    const size_t row_bytes = (size_t)s.I * 2;
    const long long total = (long long)T * s.H;
    for (long long item = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5); item < total;
         item += (long long)gridDim.x * kWarps) {
        const int t = (int)(item / s.H);
        const int m = (int)(item - (long long)t * s.H);
        float acc = 0.f;
        for (int j0 = 0; j0 < s.k; j0 += JB) {
            int4 wv[JB][CPL];
            bool act[JB];
#pragma unroll
            for (int jj = 0; jj < JB; ++jj) {
                const int j = j0 + jj;
                const int i = t * s.k + j;
                act[jj] = j < s.k && L.entry_wave[i] == wave;
                if (act[jj]) {
                    const uint8_t* row = slots + (size_t)L.entry_slot[i] * s.stride + s.w2_off +
                                         (size_t)m * row_bytes;
#pragma unroll
                    for (int c = 0; c < CPL; ++c) {
                        const int idx = lane + 32 * c;
                        wv[jj][c] = idx < nchunk ? ldg16(row + 16 * (size_t)idx) : make_int4(0, 0, 0, 0);
                    }
                }
            }
#pragma unroll
            for (int jj = 0; jj < JB; ++jj) {
                if (!act[jj]) continue;
                const int i = t * s.k + j0 + jj;
                const float* h = hbuf + (size_t)i * s.I;
                float d = 0.f;
#pragma unroll
                for (int c = 0; c < CPL; ++c) {
                    const int idx = lane + 32 * c;
                    if (idx < nchunk) {
                        const float4 h0 = __ldg(reinterpret_cast<const float4*>(h + 8 * idx));
                        const float4 h1 = __ldg(reinterpret_cast<const float4*>(h + 8 * idx + 4));
                        d = dot8_bf16_f32(wv[jj][c], h0, h1, d);
                    }
                }
                d = warp_sum(d);
                const float p = __fmul_rn(L.topk_w[i], d);
                if (fused)
                    acc = __fadd_rn(acc, p);
                else if (lane == 0)
                    merged[(size_t)i * s.H + m] = p;
            }
        }
        if (fused && lane == 0) out[(size_t)t * s.H + m] = __float2bfloat16_rn(acc);
    }
}

__global__ void topk_sum_kernel(const float* __restrict__ merged, __nv_bfloat16* __restrict__ out,
                                int T, int k, int H) {
    const long long total = (long long)T * H;
    for (long long q = (long long)blockIdx.x * blockDim.x + threadIdx.x; q < total;
         q += (long long)gridDim.x * blockDim.x) {
        const int t = (int)(q / H);
        const int m = (int)(q - (long long)t * H);
        float acc = 0.f;
        for (int j = 0; j < k; ++j) acc = __fadd_rn(acc, merged[((size_t)t * k + j) * H + m]);
        out[q] = __float2bfloat16_rn(acc);
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
#define PE_GATEUP(C) gateup_bf16_kernel<C><<<grid, kThreads, 0, st>>>(L, s, x, slots_layer, wave, T, hbuf)
    if (cpl <= 1) PE_GATEUP(1);
    else if (cpl <= 2) PE_GATEUP(2);
    else if (cpl <= 4) PE_GATEUP(4);
    else if (cpl <= 8) PE_GATEUP(8);
    else if (cpl <= 16) PE_GATEUP(16);
    else return cudaErrorInvalidValue;
#undef PE_GATEUP
    return cudaGetLastError();
}

cudaError_t launch_down(const LayerDev& L, const Shape& s, const uint8_t* slots_layer, int wave,
                        int T, const float* hbuf, float* merged, __nv_bfloat16* out, int fused,
                        int num_sms, cudaStream_t st) {
    const int grid = grid_for((long long)T * s.H, num_sms);
    if (grid <= 0) return cudaSuccess;
    const int cpl = (s.I / 8 + 31) / 32;
#define PE_DOWN(C) down_bf16_kernel<C><<<grid, kThreads, 0, st>>>(L, s, slots_layer, wave, T, hbuf, merged, out, fused)
    if (cpl <= 1) PE_DOWN(1);
    else if (cpl <= 2) PE_DOWN(2);
    else if (cpl <= 3) PE_DOWN(3);
    else if (cpl <= 4) PE_DOWN(4);
    else if (cpl <= 8) PE_DOWN(8);
    else return cudaErrorInvalidValue;
#undef PE_DOWN
    return cudaGetLastError();
}

cudaError_t launch_topk_sum(const Shape& s, const float* merged, __nv_bfloat16* out, int T,
                            cudaStream_t st) {
    const long long total = (long long)T * s.H;
    const int grid = (int)((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
    if (grid <= 0) return cudaSuccess;
    topk_sum_kernel<<<grid, 256, 0, st>>>(merged, out, T, s.k, s.H);
    return cudaGetLastError();
}

}  // namespace pe
