// Device-side helpers shared by the kernel files.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ssd_internal.cuh"

namespace ssd {

__device__ __forceinline__ float ld_in(const float* p, long long i) { return __ldg(p + i); }
__device__ __forceinline__ float ld_in(const __nv_bfloat16* p, long long i) {
    return __bfloat162float(p[i]);
}
__device__ __forceinline__ void st_out(float* p, long long i, float v) { p[i] = v; }
__device__ __forceinline__ void st_out(__nv_bfloat16* p, long long i, float v) {
    p[i] = __float2bfloat16_rn(v);
}
// Elements 4 i .. 4 i + 3 of p (16-byte aligned base).
__device__ __forceinline__ void st_out4(float* p, long long i, float4 v) {
    reinterpret_cast<float4*>(p)[i] = v;
}
__device__ __forceinline__ void st_out4(__nv_bfloat16* p, long long i, float4 v) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
    reinterpret_cast<uint2*>(p)[i] =
        make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
}

// delta = softplus(raw + delta_init): log(1 + e^z) written without overflow.
__device__ __forceinline__ float softplus_f(float z) {
    return fmaxf(z, 0.f) + log1pf(expf(-fabsf(z)));
}
// d softplus / dz
__device__ __forceinline__ float sigmoid_f(float z) { return 1.f / (1.f + expf(-z)); }

// Records the first device-side error; later ones are dropped.
__device__ __forceinline__ void set_status(WsHeader* h, int code) {
    atomicCAS(&h->status, 0, code);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

}  // namespace ssd
