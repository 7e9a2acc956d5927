// Device helpers shared by the streaming kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace pe {

// 16-byte load that bypasses L1 (host-store rows are read once per page-in).
__device__ __forceinline__ int4 ld_nc_na(const void* p) {
    int4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.s32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// 16-byte read-only load (weights in slots, activations).
__device__ __forceinline__ int4 ldg16(const void* p) { return __ldg(reinterpret_cast<const int4*>(p)); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// c + a * b for bf16 a, b (the low or high halves of two 32-bit registers)
// with one rounding to fp32: the mixed-precision fma of sm_100 and later,
// equal to fmaf(float(a), float(b), c).
__device__ __forceinline__ float fma_bf16_lo(uint32_t a, uint32_t b, float c) {
    float d;
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, al, bl, %3;\n\t}"
        : "=f"(d)
        : "r"(a), "r"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float fma_bf16_hl(uint32_t a, uint32_t b, float c) {  // a high, b low
    float d;
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, ah, bl, %3;\n\t}"
        : "=f"(d)
        : "r"(a), "r"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float fma_bf16_lh(uint32_t a, uint32_t b, float c) {  // a low, b high
    float d;
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, al, bh, %3;\n\t}"
        : "=f"(d)
        : "r"(a), "r"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float fma_bf16_hh(uint32_t a, uint32_t b, float c) {
    float d;
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, ah, bh, %3;\n\t}"
        : "=f"(d)
        : "r"(a), "r"(b), "f"(c));
    return d;
}

// Totals over the warp of R per-lane values (R rows), by a transposed
// butterfly: at each of the first log2(R) steps (lane distance 16, 8, ...) a
// lane keeps half of the rows it holds, adds its partner's copy of them and
// hands the other half to the partner, then the usual butterfly finishes.
// Every row's total is formed by the same tree of additions as warp_sum (so
// the same value, bit for bit) with R - 1 + 5 - log2(R) shuffles instead of
// 5R.  Lane l returns the total of row (l >> (5 - log2 R)) & (R - 1).
template <int R>
__device__ __forceinline__ float warp_sum_rows(float (&v)[R], int lane) {
    static_assert(R == 1 || R == 2 || R == 4 || R == 8, "1, 2, 4 or 8 rows");
    constexpr int LOGR = R == 8 ? 3 : R == 4 ? 2 : R == 2 ? 1 : 0;
#pragma unroll
    for (int step = 0; step < LOGR; ++step) {
        const int o = 16 >> step, n = R >> step;  // rows held before this step
        const bool hi = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float keep = hi ? v[i + n / 2] : v[i];
            const float send = hi ? v[i] : v[i + n / 2];
            v[i] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, o));
        }
    }
    float t = v[0];
#pragma unroll
    for (int o = 16 >> LOGR; o; o >>= 1) t = __fadd_rn(t, __shfl_xor_sync(0xffffffffu, t, o));
    return t;
}

// acc += sum of the 8 bf16 products of w and x, in element order, each
// through the mixed-precision fma (the same value as fmaf on the operands
// widened to fp32).
__device__ __forceinline__ float dot8_bf16(int4 w, int4 x, float acc) {
    const uint32_t wv[4] = {(uint32_t)w.x, (uint32_t)w.y, (uint32_t)w.z, (uint32_t)w.w};
    const uint32_t xv[4] = {(uint32_t)x.x, (uint32_t)x.y, (uint32_t)x.z, (uint32_t)x.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        acc = fma_bf16_lo(wv[q], xv[q], acc);
        acc = fma_bf16_hh(wv[q], xv[q], acc);
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

__device__ __forceinline__ float silu(float g) { return __fdiv_rn(g, __fadd_rn(1.f, expf(-g))); }

// h = SiLU(gate . x) * (up . x) for one gate/up row pair held by the warp
// (chunk c of lane l covers elements 8*(l + 32c) .. +7).  Every path that
// computes an h value goes through this function, so h does not depend on
// where the weights were read from.
// xr is a generic pointer to the token's bf16 row (shared or global memory).
template <int CPL>
__device__ __forceinline__ float row_pair_h(const int4 (&gv)[CPL], const int4 (&uv)[CPL], const uint8_t* xr,
                                            int lane, int nchunk) {
    float ag = 0.f, au = 0.f;
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
        const int idx = lane + 32 * c;
        const int4 xv = idx < nchunk ? *reinterpret_cast<const int4*>(xr + 16 * (size_t)idx) : make_int4(0, 0, 0, 0);
        ag = dot8_bf16(gv[c], xv, ag);
        au = dot8_bf16(uv[c], xv, au);
    }
    ag = warp_sum(ag);
    au = warp_sum(au);
    return __fmul_rn(silu(ag), au);
}

}  // namespace pe

namespace pe {

// Programmatic dependent launch.  Kernels launched through launch_pdl may
// start while the previous kernel on the stream is still running; each of
// them calls pdl_wait() before touching anything the previous kernel writes
// (it returns once that kernel has completed and its writes are visible),
// and pdl_trigger() to let the next kernel start early.  Without the launch
// attribute both are no-ops.
// Position of float4 v of chunk idx (F4 float4s per chunk, one chunk per
// lane) in an h vector staged in shared memory: the float4s of each chunk are
// XOR-swizzled by the chunk index so that the eight lanes of a quarter warp,
// reading the same v of eight consecutive chunks, hit eight different 16-byte
// bank groups.
template <int F4>
__device__ __forceinline__ int hs_pos(int idx, int v) {
    static_assert(F4 == 2 || F4 == 4 || F4 == 8, "chunks of 8, 16 or 32 h values");
    if constexpr (F4 == 8) return idx * 8 + (v ^ (idx & 7));
    else if constexpr (F4 == 4) return idx * 4 + (v ^ ((idx >> 1) & 3));
    else return idx * 2 + (v ^ ((idx >> 2) & 1));
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace pe
