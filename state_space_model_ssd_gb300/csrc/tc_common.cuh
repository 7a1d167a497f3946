// Shared pieces of the tensor-core kernels: tile constants, tensor-map
// encoding (host), bounded waits with cooperative abort, bf16 helpers.
#pragma once

#include <mutex>

#include "ssd_device.cuh"
#include "tc_ptx.cuh"

namespace ssd {
namespace tcc {

using namespace tc;

constexpr int kQ = 64;                 // chunk length
constexpr int kP = 64;                 // head dimension
// Largest delta sum over a chunk that the factorisation exp(s_t - s_s) = f(t) g(s) / delta_s
// carries: factors stay within exp(+-64).  Chunks beyond it run the SIMT evaluation.
constexpr float kMaxChunkDecay = 128.f;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint32_t kSleepHintNs = 20000;  // longest suspension per check of a wait

// ---------------------------------------------------------------- host: tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 3-D bf16 map over a [T][D1][D0] tensor, dims ordered (D0, D1, T), box
// (64, 1, 64): one 64 x 64 tile of one head (or group) per copy.
inline bool make_map(CUtensorMap* m, const void* base, long long T, int D1, int D0) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D0, (cuuint64_t)D1, (cuuint64_t)T};
    cuuint64_t strides[2] = {(cuuint64_t)D0 * 2, (cuuint64_t)D1 * D0 * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
               box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D fp32 map over a [T][D1][D0] tensor, dims (D0, D1, T), box (32, 1, 64):
// one 64-row x 128-byte tile (128-byte swizzle), used to add partial dB/dC tiles.
inline bool make_map_f32(CUtensorMap* m, const void* base, long long T, int D1, int D0) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D0, (cuuint64_t)D1, (cuuint64_t)T};
    cuuint64_t strides[2] = {(cuuint64_t)D0 * 4, (cuuint64_t)D1 * D0 * 4};
    cuuint32_t box[3] = {32, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---------------------------------------------------------------- device helpers
__device__ __forceinline__ void named_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Bounded wait that also gives up as soon as another thread has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity,
                                              volatile int* abort_flag, WsHeader* hdr) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        // suspended in hardware between checks (woken when the phase completes)
        if (mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > kWaitNs) {
            *abort_flag = 1;
            set_status(hdr, SSD_ERR_TIMEOUT);
            return false;
        }
    }
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
}

// s * (16 fp32 values) as 16 bf16 (32 bytes) at p: one 256-bit store when wide (p 32-byte
// aligned), else two 128-bit stores.  A warp whose lanes write different rows then fills
// whole 32-byte sectors with each store.
__device__ __forceinline__ void store_bf16x16(void* p, const uint32_t* v, float s, bool wide) {
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        w[i] = pack_bf16(s * __uint_as_float(v[2 * i]), s * __uint_as_float(v[2 * i + 1]));
    if (wide) {
        asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p),
                     "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]),
                     "r"(w[7])
                     : "memory");
    } else {
        reinterpret_cast<uint4*>(p)[0] = make_uint4(w[0], w[1], w[2], w[3]);
        reinterpret_cast<uint4*>(p)[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
}

// Multiplies the 8 bf16 values of a 16-byte chunk by s.
__device__ __forceinline__ uint4 scale_chunk(uint4 v, float s) {
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&w[i]);
        float2 f = __bfloat1622float2(b);
        w[i] = pack_bf16(f.x * s, f.y * s);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Inclusive prefix sum within a warp.
__device__ __forceinline__ float warp_scan(float v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    return v;
}


}  // namespace tcc
}  // namespace ssd
