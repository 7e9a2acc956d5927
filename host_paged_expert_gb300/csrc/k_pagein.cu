// Page-in: copy the experts a wave planned from the host store into slots.
//
// "Paged Experts" (SGLang docs), "Captured decode".  The copy is done by
// GPU threads that load the host store's rows directly (the store is pinned
// and mapped, so it has a device-visible address); how many rows to move is
// read from the plan in device memory, so a replayed graph copies whatever
// that replay's plan chose, with no host involvement.  One expert row holds
// all of an expert's paged tensors (w13, w2 and any scale tensors), so one
// row copy moves them together and a slot never pairs one expert's weights
// with another expert's scales.
//
// The grid is fixed from shapes (a few CTAs per SM); CTAs stride over
// (planned expert, 16 KiB chunk) items and stop at the device-side count.

#include "pe_device.cuh"
#include "pe_internal.h"

namespace pe {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;
constexpr size_t kChunk = (size_t)kCopyThreads * 16 * kCopyUnroll;  // bytes per item

// Copy one chunk of up to kChunk bytes (a multiple of 16).
__device__ __forceinline__ void copy_chunk(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                           size_t bytes) {
    const int4* s = reinterpret_cast<const int4*>(src);
    int4* d = reinterpret_cast<int4*>(dst);
    const int nvec = (int)(bytes >> 4);
    int4 v[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
        const int i = threadIdx.x + u * kCopyThreads;
        if (i < nvec) v[u] = ld_nc_na(s + i);
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
        const int i = threadIdx.x + u * kCopyThreads;
        if (i < nvec) d[i] = v[u];
    }
}

__global__ void __launch_bounds__(kCopyThreads) pagein_kernel(
    const uint8_t* __restrict__ host_layer, uint8_t* __restrict__ slots_layer, size_t stride,
    size_t copy_bytes, const int32_t* __restrict__ plan_expert, const int32_t* __restrict__ plan_slot,
    const int32_t* __restrict__ plan_count, int max_count) {
    pdl_wait();
    pdl_trigger();
    const int count = min(*plan_count, max_count);
    const size_t nchunk = (copy_bytes + kChunk - 1) / kChunk;
    const size_t items = (size_t)count * nchunk;
    for (size_t it = blockIdx.x; it < items; it += gridDim.x) {
        const int p = (int)(it / nchunk);
        const size_t c = it - (size_t)p * nchunk;
        const size_t off = c * kChunk;
        const size_t e = (size_t)plan_expert[p];
        const size_t slot = (size_t)plan_slot[p];
        copy_chunk(host_layer + e * stride + off, slots_layer + slot * stride + off,
                   min(kChunk, copy_bytes - off));
    }
}

__global__ void __launch_bounds__(kCopyThreads) copy_kernel(const uint8_t* __restrict__ src,
                                                            uint8_t* __restrict__ dst, size_t bytes) {
    const size_t nchunk = (bytes + kChunk - 1) / kChunk;
    for (size_t c = blockIdx.x; c < nchunk; c += gridDim.x) {
        const size_t off = c * kChunk;
        copy_chunk(src + off, dst + off, min(kChunk, bytes - off));
    }
}

}  // namespace

cudaError_t launch_pagein(const LayerDev& L, const Shape& s, const uint8_t* host_layer,
                          uint8_t* slots_layer, int wave, int max_count, int num_sms,
                          cudaStream_t st) {
    const size_t nchunk = (s.copy_bytes + kChunk - 1) / kChunk;
    const size_t want = (size_t)max_count * nchunk;
    const int grid = (int)min(want, (size_t)num_sms * 4);
    if (grid <= 0) return cudaSuccess;
    return launch_pdl(pagein_kernel, grid, kCopyThreads, 0, st, host_layer, slots_layer, s.stride, s.copy_bytes,
                      (const int32_t*)(L.plan_expert + (size_t)wave * s.K),
                      (const int32_t*)(L.plan_slot + (size_t)wave * s.K), (const int32_t*)(L.plan_count + wave),
                      max_count);
}

cudaError_t launch_copy(const void* src, void* dst, size_t bytes, int num_sms, cudaStream_t st) {
    const size_t nchunk = (bytes + kChunk - 1) / kChunk;
    const int grid = (int)min(nchunk, (size_t)num_sms * 4);
    if (grid <= 0) return cudaSuccess;
    copy_kernel<<<grid, kCopyThreads, 0, st>>>((const uint8_t*)src, (uint8_t*)dst, bytes);
    return cudaGetLastError();
}

}  // namespace pe
