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

}  // namespace pe
