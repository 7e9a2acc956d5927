// One expert's SiLU-gated MLP with its scratch in a static device array.
//
// Some callers cannot allocate device memory at the point where they need
// this computation: code running under a framework that hands out all device
// memory itself (a plugin that may only use the buffers it is given), code on
// a path that must never grow its memory footprint, or code in a context
// where calling cudaMalloc would synchronise the device.  For them,
// pe_expert_mlp_noalloc computes out[t] = down . (SiLU(gate . x_t) * (up . x_t))
// for one bf16 expert without allocating anything: the intermediate h lives
// in g_mlp_scratch, a file-scope device array that every GPU loading this
// library holds until the process exits.
//
// The arithmetic is the same device code as the decode path of pe_forward
// (the same row_pair_h and down-row dot product, fp32 accumulation, one
// rounding to bf16 at the end), so a one-expert layer (E = K = top_k = 1,
// router weight exactly 1) gives the same result through either entry point.

#include <mutex>

#include "pe_device.cuh"
#include "pe_internal.h"

namespace pe {
namespace {

constexpr size_t kScratchFloats = PE_NOALLOC_SCRATCH_BYTES / sizeof(float);
constexpr int kMaxDevices = 64;
constexpr int kThreadsNA = 256;
constexpr int kWarpsNA = kThreadsNA / 32;

// h[t, n] for all tokens of the call.  Every element a call reads is written
// earlier in the same call, so nothing needs clearing between calls.
static __device__ __align__(256) float g_mlp_scratch[kScratchFloats];

std::mutex g_mu;
float* g_scratch_ptr[kMaxDevices] = {};  // device address of g_mlp_scratch, per device

// h[t, n] = SiLU(gate_n . x_t) * (up_n . x_t): one warp per (t, n).
template <int CPL>
__global__ void __launch_bounds__(kThreadsNA) noalloc_gateup_kernel(const uint8_t* __restrict__ w13,
                                                                    const uint8_t* __restrict__ x,
                                                                    float* __restrict__ h, int T, int H,
                                                                    int I) {
    const int lane = threadIdx.x & 31;
    const int nchunk = H >> 3;
    const size_t row_bytes = (size_t)H * 2;
    const long long total = (long long)T * I;
    for (long long item = (long long)blockIdx.x * kWarpsNA + (threadIdx.x >> 5); item < total;
         item += (long long)gridDim.x * kWarpsNA) {
        const int t = (int)(item / I);
        const int n = (int)(item - (long long)t * I);
        const uint8_t* g = w13 + (size_t)n * row_bytes;
        const uint8_t* u = w13 + (size_t)(I + n) * row_bytes;
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
        const float hv = row_pair_h<CPL>(gv, uv, x + (size_t)t * row_bytes, lane, nchunk);
        if (lane == 0) h[(size_t)t * I + n] = hv;
    }
}

// out[t, m] = bf16(down_m . h_t): one warp per (t, m).
template <int CPL>
__global__ void __launch_bounds__(kThreadsNA) noalloc_down_kernel(const uint8_t* __restrict__ w2,
                                                                  const float* __restrict__ h,
                                                                  __nv_bfloat16* __restrict__ out, int T,
                                                                  int H, int I) {
    const int lane = threadIdx.x & 31;
    const int nchunk = I >> 3;
    const size_t row_bytes = (size_t)I * 2;
    const long long total = (long long)T * H;
    for (long long item = (long long)blockIdx.x * kWarpsNA + (threadIdx.x >> 5); item < total;
         item += (long long)gridDim.x * kWarpsNA) {
        const int t = (int)(item / H);
        const int m = (int)(item - (long long)t * H);
        const uint8_t* row = w2 + (size_t)m * row_bytes;
        const float* ht = h + (size_t)t * I;
        float d = 0.f;
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            const int idx = lane + 32 * c;
            if (idx < nchunk) {
                const int4 wv = ldg16(row + 16 * (size_t)idx);
                const float4 h0 = __ldg(reinterpret_cast<const float4*>(ht + 8 * idx));
                const float4 h1 = __ldg(reinterpret_cast<const float4*>(ht + 8 * idx + 4));
                d = dot8_bf16_f32(wv, h0, h1, d);
            }
        }
        d = warp_sum(d);
        // router weight 1 and a one-entry top-k sum, as in the decode path
        if (lane == 0) out[(size_t)t * H + m] = __float2bfloat16_rn(__fadd_rn(0.f, __fmul_rn(1.f, d)));
    }
}

// Device address of g_mlp_scratch on the current device, looked up once per
// device with that device current.
cudaError_t scratch_for_current_device(float** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_mlp_scratch);
        if (e) return e;
        g_scratch_ptr[dev] = static_cast<float*>(p);
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace pe

using namespace pe;

extern "C" pe_status pe_expert_mlp_noalloc(const void* w13, const void* w2, const void* x, void* out,
                                           int32_t num_tokens, int32_t hidden, int32_t intermediate,
                                           void* stream) {
    if (!w13 || !w2 || !x || !out) {
        set_thread_error("pe_expert_mlp_noalloc: NULL pointer");
        return PE_ERR_INVALID;
    }
    const uintptr_t al = reinterpret_cast<uintptr_t>(w13) | reinterpret_cast<uintptr_t>(w2) |
                         reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(out);
    if (al % 16) {
        set_thread_error("pe_expert_mlp_noalloc: pointers must be 16-byte aligned");
        return PE_ERR_INVALID;
    }
    if (num_tokens < 0 || hidden < 8 || hidden % 8 || intermediate < 8 || intermediate % 8) {
        set_thread_error("pe_expert_mlp_noalloc: hidden and intermediate must be positive multiples of 8");
        return PE_ERR_INVALID;
    }
    if (hidden > 2048 || intermediate > 1024) {
        set_thread_error("pe_expert_mlp_noalloc: hidden above 2048 or intermediate above 1024");
        return PE_ERR_RANGE;
    }
    if ((size_t)num_tokens * (size_t)intermediate * sizeof(float) > PE_NOALLOC_SCRATCH_BYTES) {
        set_thread_error("pe_expert_mlp_noalloc: num_tokens * intermediate * 4 exceeds PE_NOALLOC_SCRATCH_BYTES");
        return PE_ERR_RANGE;
    }
    if (num_tokens == 0) return PE_OK;
    float* h = nullptr;
    cudaError_t e = scratch_for_current_device(&h);
    if (e) {
        set_thread_error(cudaGetErrorString(e));
        return PE_ERR_CUDA;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const auto* w13b = static_cast<const uint8_t*>(w13);
    const auto* w2b = static_cast<const uint8_t*>(w2);
    const auto* xb = static_cast<const uint8_t*>(x);
    auto* y = static_cast<__nv_bfloat16*>(out);
    const int T = num_tokens, H = hidden, I = intermediate;
    auto grid = [](long long warps) {
        const long long b = (warps + kWarpsNA - 1) / kWarpsNA;
        return (int)(b < 4096 ? b : 4096);
    };
    const int cph = (H / 8 + 31) / 32, cpi = (I / 8 + 31) / 32;
    const int g1 = grid((long long)T * I), g2 = grid((long long)T * H);
    if (cph <= 1) noalloc_gateup_kernel<1><<<g1, kThreadsNA, 0, st>>>(w13b, xb, h, T, H, I);
    else if (cph <= 2) noalloc_gateup_kernel<2><<<g1, kThreadsNA, 0, st>>>(w13b, xb, h, T, H, I);
    else if (cph <= 4) noalloc_gateup_kernel<4><<<g1, kThreadsNA, 0, st>>>(w13b, xb, h, T, H, I);
    else noalloc_gateup_kernel<8><<<g1, kThreadsNA, 0, st>>>(w13b, xb, h, T, H, I);
    e = cudaGetLastError();
    if (!e) {
        if (cpi <= 1) noalloc_down_kernel<1><<<g2, kThreadsNA, 0, st>>>(w2b, h, y, T, H, I);
        else if (cpi <= 2) noalloc_down_kernel<2><<<g2, kThreadsNA, 0, st>>>(w2b, h, y, T, H, I);
        else if (cpi <= 3) noalloc_down_kernel<3><<<g2, kThreadsNA, 0, st>>>(w2b, h, y, T, H, I);
        else noalloc_down_kernel<4><<<g2, kThreadsNA, 0, st>>>(w2b, h, y, T, H, I);
        e = cudaGetLastError();
    }
    if (e) {
        set_thread_error(cudaGetErrorString(e));
        return PE_ERR_CUDA;
    }
    return PE_OK;
}
