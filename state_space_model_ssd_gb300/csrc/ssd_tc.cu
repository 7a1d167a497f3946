// Tensor-core path: bf16 x/B/C, P = 64, N in {64, 128}, chunk Q = 64, two heads
// of one B/C group per CTA.
//
// Every dense contraction of the chunked (semiseparable) form of page "长序列
// Mamba 多卡训练算力和显存怎么同时省" §一 runs on tcgen05 with fp32 accumulators in
// TMEM, operands staged by TMA in 128-byte-swizzled shared memory:
//
//   per chunk c (tokens t, s in c; chunk-local log-decay s_t = -sum_{k<=t} delta_k,
//   reference point m = s_end / 2, f(t) = exp(s_t - m), g(s) = delta_s exp(m - s_s)):
//     G1  CB[t, s]       = C_t . B_s                                  (M=64,  N=64,  K=N)
//     L0[t, s]           = CB[t, s] * [s <= t]                      (epilogue, bf16)
//     G2  Y[(h,p), t]    = sum_s g(s) x_s[(h,p)] L0[t, s]            (M=128, N=64,  K=64)
//     G3  Y[(h,p), t]   += sum_n exp(m) H[(h,p), n] C_t[n]           (M=128, N=64,  K=N)
//         y_t            = f(t) Y[., t]            = diagonal block + exp(s_t) H C_t
//     G4  S[(h,p), n]    = sum_s g(s) x_s[(h,p)] B_s[n]              (M=128, N=N,   K=64)
//         H             <- exp(s_end) H + exp(s_end - m) S          (fp32, registers)
//
// The factorisation exp(s_t - s_s) = f(t) g(s) / delta_s keeps every exponent in
// [-|s_end|/2, |s_end|/2]; chunks whose delta sum exceeds kMaxChunkDecay would
// leave fp32 range and are reported through the status word.
//
// tc_fwd_state computes the segment aggregates sum_t exp(Lambda_end - Lambda_t)
// delta_t x_t B_t^T (the G4 contraction over a whole segment) for the scan in
// ssd_scan.cu; tc_fwd_walk then walks each segment chunk by chunk from the state
// entering it.
#include <mutex>

#include "ssd_device.cuh"
#include "tc_ptx.cuh"

namespace ssd {

using namespace tc;

namespace {

constexpr int kQ = 64;                 // chunk length
constexpr int kP = 64;                 // head dimension
constexpr float kMaxChunkDecay = 160.f;
constexpr uint64_t kWaitNs = 2000000000ull;

// ---------------------------------------------------------------- host: tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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
bool make_map(CUtensorMap* m, const void* base, long long T, int D1, int D0) {
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

// ---------------------------------------------------------------- device helpers
__device__ __forceinline__ void named_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Bounded wait that also gives up as soon as another thread has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity,
                                              volatile int* abort_flag, WsHeader* hdr) {
    if (*abort_flag) return false;
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
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

// ================================================================ segment aggregates
// Warps: 0 = TMA producer, 1 = MMA issuer (and TMEM owner), 2..5 = compute.
constexpr int kStateStages = 4;
constexpr int kStateThreads = 192;
constexpr int kMaxSeg = 1024;  // segment length bound for the per-token weights

struct StateSmem {
    // stage = X h0 (8K) | X h1 (8K) | B (N/64 x 8K)
    static constexpr int stage_bytes(int N) { return 16384 + N * 128; }
};

template <int N>
__global__ void __launch_bounds__(kStateThreads, 1)
    tc_fwd_state_kernel(const __grid_constant__ CUtensorMap map_x,
                        const __grid_constant__ CUtensorMap map_b, Args a) {
    const int seg = blockIdx.x;
    const int h0 = blockIdx.y * 2;
    if (seg >= a.hdr->nseg) return;
    const SegInfo si = a.segtab[seg];
    const int g = h0 / (a.H / a.G);
    const int nchunks = (si.len + kQ - 1) / kQ;
    constexpr int SB = StateSmem::stage_bytes(N);

    extern __shared__ __align__(1024) unsigned char smraw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smraw) + 1023) & ~(uintptr_t)1023);
    unsigned char* stages = sm;
    float* wts = reinterpret_cast<float*>(sm + kStateStages * SB);   // [2][kMaxSeg]
    float* red = wts + 2 * kMaxSeg;                                 // [8]
    uint64_t* full = reinterpret_cast<uint64_t*>(red + 8);
    uint64_t* empty = full + kStateStages;
    uint64_t* ready = empty + kStateStages;
    uint64_t* done = ready + kStateStages;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int i = 0; i < kStateStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
            mbar_init(&ready[i], 128);
        }
        mbar_init(done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tslot, N);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == 0) {
        if (lane == 0) {
            for (int c = 0; c < nchunks; ++c) {
                const int s = c % kStateStages;
                if (c >= kStateStages &&
                    !wait_or_abort(&empty[s], ((c / kStateStages) - 1) & 1, abort_flag, a.hdr))
                    break;
                unsigned char* st = stages + s * SB;
                const int tok = (int)(si.start + (long long)c * kQ);
                mbar_expect_tx(&full[s], SB);
                tma_load_3d(st, &map_x, &full[s], 0, h0, tok);
                tma_load_3d(st + 8192, &map_x, &full[s], 0, h0 + 1, tok);
                for (int nb = 0; nb < N / 64; ++nb)
                    tma_load_3d(st + 16384 + nb * 8192, &map_b, &full[s], nb * 64, g, tok);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(128, N, 1, 1);
            for (int c = 0; c < nchunks; ++c) {
                const int s = c % kStateStages;
                if (!wait_or_abort(&ready[s], (c / kStateStages) & 1, abort_flag, a.hdr)) break;
                tc_fence_after();
                const uint32_t xs = smem_u32(stages + s * SB);
                const uint32_t bs = xs + 16384;
#pragma unroll
                for (int k = 0; k < kQ / 16; ++k) {
                    const uint64_t ad = sw128_desc(xs + k * 2048, 8192, 1024);
                    const uint64_t bd = sw128_desc(bs + k * 2048, 8192, 1024);
                    mma_bf16(tmem, ad, bd, idesc, (c > 0 || k > 0) ? 1u : 0u);
                }
                mma_commit(&empty[s]);
            }
            mma_commit(done);
        }
    } else {
        // ---- compute warps: per-token weights relative to the segment end
        const int ct = tid - 64;            // 0..127
        const int head = ct >> 6;           // 0..1
        const int j = ct & 63;              // 64 threads per head
        const int per = (si.len + 63) / 64; // consecutive tokens per thread
        const int t_lo = j * per;
        float loc = 0.f;
        for (int i = 0; i < per; ++i) {
            const int t = t_lo + i;
            float d = 0.f;
            if (t < si.len)
                d = softplus_f(a.raw[(si.start + t) * a.H + h0 + head] + a.delta_init);
            loc += d;
            if (t < kMaxSeg) wts[head * kMaxSeg + t] = d;
        }
        // exclusive prefix of the per-thread sums across the head's 64 threads
        float inc = warp_scan(loc, lane);
        const int hw = (ct >> 5) & 1;  // warp within the head
        if (lane == 31) red[head * 2 + hw] = inc;
        named_sync(1, 128);
        float excl = inc - loc + (hw ? red[head * 2] : 0.f);
        const float total = red[head * 2] + red[head * 2 + 1];
        // w_t = delta_t exp(-(sum of delta over (t, end]))
        float run = excl;
        for (int i = 0; i < per; ++i) {
            const int t = t_lo + i;
            if (t < si.len) {
                const float d = wts[head * kMaxSeg + t];
                run += d;
                wts[head * kMaxSeg + t] = d * expf(run - total);
            } else if (t < kMaxSeg) {
                wts[head * kMaxSeg + t] = 0.f;
            }
        }
        if (j == 0) a.lam[(long long)seg * a.H + h0 + head] = -total;
        named_sync(1, 128);
        // ---- scale x by the weights in place, chunk by chunk
        for (int c = 0; c < nchunks; ++c) {
            const int s = c % kStateStages;
            if (!wait_or_abort(&full[s], (c / kStateStages) & 1, abort_flag, a.hdr)) break;
            uint4* xs = reinterpret_cast<uint4*>(stages + s * SB);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int idx = ct + 128 * i;  // 0..1023 16-byte chunks of the two x tiles
                const int hh = idx >> 9;
                const int row = (idx & 511) >> 3;
                const int t = c * kQ + row;
                const float w = (t < si.len) ? wts[hh * kMaxSeg + t] : 0.f;
                xs[idx] = scale_chunk(xs[idx], w);
            }
            fence_proxy_async();
            mbar_arrive(&ready[s]);
        }
        // ---- epilogue: TMEM -> aggregates A[seg][h][p][n]
        const bool ok = wait_or_abort(done, 0, abort_flag, a.hdr);
        tc_fence_after();
        const int q = warp & 3;
        const int r = 32 * q + lane;  // accumulator row = (head, p)
        float* Arow = a.A + (((long long)seg * a.H + h0 + (r >> 6)) * kP + (r & 63)) * N;
#pragma unroll
        for (int c0 = 0; c0 < N; c0 += 16) {
            uint32_t v[16];
            tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + c0, v);
            tmem_wait_ld();
            if (ok) {
#pragma unroll
                for (int i = 0; i < 16; i += 4)
                    *reinterpret_cast<float4*>(Arow + c0 + i) =
                        make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                                    __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, N);
}

// ================================================================ chunk walk
// Warps: 0 = TMA producer, 1 = MMA issuer, 2..9 = compute (two warpgroups:
// WG0 = warps 2..5, WG1 = warps 6..9; each covers the 128 TMEM lanes once).
constexpr int kWalkThreads = 320;
constexpr int kCT = 256;  // compute threads

template <int N>
struct WalkLayout {
    static constexpr int STAGE = 16384 + 2 * N * 128;  // X h0 | X h1 | B | C
    static constexpr int OFF_STAGE = 0;
    static constexpr int OFF_L0 = 2 * STAGE;                 // 2 x 8K
    static constexpr int OFF_H = OFF_L0 + 2 * 8192;         // 2 x (N/64) x 16K
    static constexpr int HBUF = (N / 64) * 16384;
    static constexpr int OFF_Y = OFF_H + 2 * HBUF;          // 2 x 16K
    static constexpr int OFF_F = OFF_Y + 2 * 16384;         // f,g: [2 buf][2 head][64] x 2
    static constexpr int OFF_SC = OFF_F + 2 * 2 * 2 * 64 * 4;  // scalars [2 buf][2 head][4]
    static constexpr int OFF_RED = OFF_SC + 2 * 2 * 4 * 4;     // [8]
    static constexpr int OFF_BAR = OFF_RED + 64;
    static constexpr int NBAR = 2 * 11;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int TOTAL = OFF_MISC + 16 + 1024;  // + alignment slack
};

// TMEM columns: D1 (CB^T) 2 x 64 | Y 2 x 64 | S 2 x N
__device__ __forceinline__ uint32_t col_d1(int b) { return b * 64; }
__device__ __forceinline__ uint32_t col_y(int b) { return 128 + b * 64; }
template <int N>
__device__ __forceinline__ uint32_t col_s(int b) { return 256 + b * N; }

template <int N>
__global__ void __launch_bounds__(kWalkThreads, 1)
    tc_fwd_walk_kernel(const __grid_constant__ CUtensorMap map_x,
                       const __grid_constant__ CUtensorMap map_b,
                       const __grid_constant__ CUtensorMap map_c,
                       const __grid_constant__ CUtensorMap map_y, Args a) {
    using Lay = WalkLayout<N>;
    const int seg = blockIdx.x;
    const int h0 = blockIdx.y * 2;
    if (seg >= a.hdr->nseg) return;
    const SegInfo si = a.segtab[seg];
    const int g = h0 / (a.H / a.G);
    const int nchunks = (si.len + kQ - 1) / kQ;

    extern __shared__ __align__(1024) unsigned char smraw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smraw) + 1023) & ~(uintptr_t)1023);
    float* fbuf = reinterpret_cast<float*>(sm + Lay::OFF_F);   // [buf][head][64]
    float* gbuf = fbuf + 2 * 2 * 64;                           // [buf][head][64]
    float* scal = reinterpret_cast<float*>(sm + Lay::OFF_SC);  // [buf][head][4]: e_end, k, hs, -
    float* red = reinterpret_cast<float*>(sm + Lay::OFF_RED);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Lay::OFF_BAR);
    uint64_t* full = bars + 0;       // [2] TMA stage landed
    uint64_t* empty = bars + 2;      // [2] stage consumed by the MMAs
    uint64_t* d1_full = bars + 4;    // [2]
    uint64_t* xg_ready = bars + 6;   // [2]
    uint64_t* l0_ready = bars + 8;   // [2]
    uint64_t* s_full = bars + 10;    // [2]
    uint64_t* s_free = bars + 12;    // [2]
    uint64_t* y_full = bars + 14;    // [2]
    uint64_t* y_free = bars + 16;    // [2]
    uint64_t* h_ready = bars + 18;   // [2]
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + Lay::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
            mbar_init(&d1_full[i], 1);
            mbar_init(&xg_ready[i], kCT);
            mbar_init(&l0_ready[i], 64);
            mbar_init(&s_full[i], 1);
            mbar_init(&s_free[i], kCT);
            mbar_init(&y_full[i], 1);
            mbar_init(&y_free[i], kCT);
            mbar_init(&h_ready[i], kCT);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            for (int c = 0; c < nchunks; ++c) {
                const int s = c & 1;
                if (c >= 2 && !wait_or_abort(&empty[s], ((c >> 1) - 1) & 1, abort_flag, a.hdr))
                    break;
                unsigned char* st = sm + Lay::OFF_STAGE + s * Lay::STAGE;
                const int tok = (int)(si.start + (long long)c * kQ);
                mbar_expect_tx(&full[s], Lay::STAGE);
                tma_load_3d(st, &map_x, &full[s], 0, h0, tok);
                tma_load_3d(st + 8192, &map_x, &full[s], 0, h0 + 1, tok);
                for (int nb = 0; nb < N / 64; ++nb) {
                    tma_load_3d(st + 16384 + nb * 8192, &map_b, &full[s], nb * 64, g, tok);
                    tma_load_3d(st + 16384 + N * 128 + nb * 8192, &map_c, &full[s], nb * 64, g,
                                tok);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t id_cb = idesc_bf16(64, 64, 0, 0);
            const uint32_t id_y = idesc_bf16(128, 64, 1, 0);
            const uint32_t id_h = idesc_bf16(128, 64, 0, 0);
            const uint32_t id_s = idesc_bf16(128, N, 1, 1);
            for (int c = 0; c < nchunks; ++c) {
                const int s = c & 1, ph = (c >> 1) & 1;
                const bool last = (c == nchunks - 1);
                if (!wait_or_abort(&full[s], ph, abort_flag, a.hdr)) break;
                tc_fence_after();
                const uint32_t xs = smem_u32(sm + Lay::OFF_STAGE + s * Lay::STAGE);
                const uint32_t bs = xs + 16384;
                const uint32_t cs = bs + N * 128;
                // G1: CB^T (M = 64 rows t, N = 64 columns s, K = N)
#pragma unroll
                for (int k = 0; k < N / 16; ++k) {
                    const uint32_t koff = (k >> 2) * 8192 + (k & 3) * 32;
                    mma_bf16(tmem + col_d1(s), sw128_desc(cs + koff, 16, 1024),
                             sw128_desc(bs + koff, 16, 1024), id_cb, k > 0 ? 1u : 0u);
                }
                mma_commit(&d1_full[s]);
                if (!wait_or_abort(&xg_ready[s], ph, abort_flag, a.hdr)) break;
                tc_fence_after();
                // G4: chunk state contribution (not needed after the last chunk)
                if (!last) {
                    if (c >= 2 && !wait_or_abort(&s_free[s], ph ^ 1, abort_flag, a.hdr)) break;
                    tc_fence_after();
#pragma unroll
                    for (int k = 0; k < kQ / 16; ++k)
                        mma_bf16(tmem + col_s<N>(s), sw128_desc(xs + k * 2048, 8192, 1024),
                                 sw128_desc(bs + k * 2048, 8192, 1024), id_s, k > 0 ? 1u : 0u);
                    mma_commit(&s_full[s]);
                }
                // G2: diagonal block
                if (!wait_or_abort(&l0_ready[s], ph, abort_flag, a.hdr)) break;
                if (c >= 2 && !wait_or_abort(&y_free[s], ph ^ 1, abort_flag, a.hdr)) break;
                tc_fence_after();
                const uint32_t l0 = smem_u32(sm + Lay::OFF_L0 + s * 8192);
#pragma unroll
                for (int k = 0; k < kQ / 16; ++k)
                    mma_bf16(tmem + col_y(s), sw128_desc(xs + k * 2048, 8192, 1024),
                             sw128_desc(l0 + k * 32, 16, 1024), id_y, k > 0 ? 1u : 0u);
                // G3: state entering the chunk
                if (!wait_or_abort(&h_ready[s], ph, abort_flag, a.hdr)) break;
                tc_fence_after();
                const uint32_t hs = smem_u32(sm + Lay::OFF_H + s * Lay::HBUF);
#pragma unroll
                for (int k = 0; k < N / 16; ++k) {
                    const uint32_t ka = (k >> 2) * 16384 + (k & 3) * 32;
                    const uint32_t kb = (k >> 2) * 8192 + (k & 3) * 32;
                    mma_bf16(tmem + col_y(s), sw128_desc(hs + ka, 16, 1024),
                             sw128_desc(cs + kb, 16, 1024), id_h, 1u);
                }
                mma_commit(&y_full[s]);
                mma_commit(&empty[s]);
            }
        }
    } else {
        // ------------------------------------------------ compute warpgroups
        const int ct = tid - 64;        // 0..255
        const int wg = ct >> 7;         // 0 or 1
        const int q = warp & 3;         // TMEM lane quadrant
        const int r = 32 * q + lane;    // accumulator row = (head, p)
        const int rh = r >> 6, rp = r & 63;
        constexpr int NH = N / 2;       // state columns per warpgroup
        const int n0 = wg * NH;
        float H[NH];

        // chunk factors for chunk cc into buffer cc & 1 (threads 0..127 compute)
        auto factors = [&](int cc) {
            named_sync(1, kCT);
            if (ct < 128) {
                const int head = ct >> 6, t = ct & 63;
                const int vc = min(kQ, si.len - cc * kQ);
                float d = 0.f;
                if (t < vc)
                    d = softplus_f(a.raw[(si.start + (long long)cc * kQ + t) * a.H + h0 + head] +
                                   a.delta_init);
                float inc = warp_scan(d, lane);
                const int hw = (ct >> 5) & 1;
                if (lane == 31) red[head * 2 + hw] = inc;
                // wait for both warps of the head (64 threads per head, ids 2 and 3)
                named_sync(2 + head, 64);
                if (hw) inc += red[head * 2];
                const float send = red[head * 2] + red[head * 2 + 1];  // sum of delta
                const float sc = -inc;            // s_t
                const float mid = -0.5f * send;   // reference point
                const int b = cc & 1;
                fbuf[(b * 2 + head) * 64 + t] = expf(sc - mid);
                gbuf[(b * 2 + head) * 64 + t] = d * expf(mid - sc);
                if (t == 0) {
                    scal[(b * 2 + head) * 4 + 0] = expf(-send);        // exp(s_end)
                    scal[(b * 2 + head) * 4 + 1] = expf(-send - mid);  // exp(s_end - m)
                    scal[(b * 2 + head) * 4 + 2] = expf(mid);          // exp(m)
                    if (send > kMaxChunkDecay) set_status(a.hdr, SSD_ERR_DEVICE);
                }
            }
            named_sync(1, kCT);
        };

        // writes bf16(H * exp(m_cc)) into the H operand buffer for chunk cc
        auto write_h = [&](int cc) {
            const int b = cc & 1;
            const float hsc = scal[(b * 2 + rh) * 4 + 2];
            unsigned char* hb = sm + Lay::OFF_H + b * Lay::HBUF;
#pragma unroll
            for (int c8 = 0; c8 < NH; c8 += 8) {
                const int n = n0 + c8;
                uint4 v = make_uint4(pack_bf16(H[c8] * hsc, H[c8 + 1] * hsc),
                                     pack_bf16(H[c8 + 2] * hsc, H[c8 + 3] * hsc),
                                     pack_bf16(H[c8 + 4] * hsc, H[c8 + 5] * hsc),
                                     pack_bf16(H[c8 + 6] * hsc, H[c8 + 7] * hsc));
                *reinterpret_cast<uint4*>(hb + (n >> 6) * 16384 + sw128_offset(r, n & 63)) = v;
            }
            fence_proxy_async();
            mbar_arrive(&h_ready[b]);
        };

        // prologue: state entering the segment, factors of chunk 0
        {
            const float* Hin = a.A + (((long long)seg * a.H + h0 + rh) * kP + rp) * N + n0;
#pragma unroll
            for (int i = 0; i < NH; i += 4) {
                const float4 v = *reinterpret_cast<const float4*>(Hin + i);
                H[i] = v.x;
                H[i + 1] = v.y;
                H[i + 2] = v.z;
                H[i + 3] = v.w;
            }
        }
        factors(0);
        write_h(0);

        for (int c = 0; c < nchunks; ++c) {
            const int s = c & 1, ph = (c >> 1) & 1;
            const bool last = (c == nchunks - 1);
            const int vc = min(kQ, si.len - c * kQ);
            const long long tok0 = si.start + (long long)c * kQ;
            unsigned char* st = sm + Lay::OFF_STAGE + s * Lay::STAGE;
            // A: x -> g(s) x in place (the operand of G2 and G4)
            const bool have = wait_or_abort(&full[s], ph, abort_flag, a.hdr);
            if (have) {
                uint4* xs = reinterpret_cast<uint4*>(st);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int idx = ct + kCT * i;  // 0..1023
                    const int hh = idx >> 9;
                    const int row = (idx & 511) >> 3;
                    xs[idx] = scale_chunk(xs[idx], gbuf[(s * 2 + hh) * 64 + row]);
                }
            }
            fence_proxy_async();
            mbar_arrive(&xg_ready[s]);
            // B: L0 = CB^T masked to s <= t (warpgroup 0, lanes 0..15 hold rows t)
            if (wg == 0) {
                const bool ok = wait_or_abort(&d1_full[s], ph, abort_flag, a.hdr);
                tc_fence_after();
                const int t = 16 * q + lane;
                unsigned char* l0 = sm + Lay::OFF_L0 + s * 8192;
#pragma unroll
                for (int c0 = 0; c0 < 64; c0 += 16) {
                    uint32_t v[16];
                    tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + col_d1(s) + c0, v);
                    tmem_wait_ld();
                    if (lane < 16 && ok) {
#pragma unroll
                        for (int e = 0; e < 16; e += 8) {
                            float f[8];
#pragma unroll
                            for (int u = 0; u < 8; ++u)
                                f[u] = (c0 + e + u <= t) ? __uint_as_float(v[e + u]) : 0.f;
                            *reinterpret_cast<uint4*>(l0 + sw128_offset(t, c0 + e)) =
                                make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]),
                                           pack_bf16(f[4], f[5]), pack_bf16(f[6], f[7]));
                        }
                    }
                }
                fence_proxy_async();
                if (lane < 16) mbar_arrive(&l0_ready[s]);
            }
            // C: state update H <- exp(s_end) H + exp(s_end - m) S
            if (!last) {
                const bool ok = wait_or_abort(&s_full[s], ph, abort_flag, a.hdr);
                tc_fence_after();
                const float e_end = scal[(s * 2 + rh) * 4 + 0];
                const float kk = scal[(s * 2 + rh) * 4 + 1];
#pragma unroll
                for (int c0 = 0; c0 < NH; c0 += 16) {
                    uint32_t v[16];
                    tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + col_s<N>(s) + n0 + c0, v);
                    tmem_wait_ld();
                    if (ok) {
#pragma unroll
                        for (int u = 0; u < 16; ++u)
                            H[c0 + u] = fmaf(e_end, H[c0 + u], kk * __uint_as_float(v[u]));
                    }
                }
                tc_fence_before();
                mbar_arrive(&s_free[s]);
                // E, F: factors of the next chunk, then its H operand
                factors(c + 1);
                write_h(c + 1);
            }
            // D: y = f(t) Y  -> staging tile -> TMA store (or direct stores on a partial chunk)
            {
                const bool ok = wait_or_abort(&y_full[s], ph, abort_flag, a.hdr);
                tc_fence_after();
                if (ct == 0) tma_store_wait_read<1>();
                named_sync(1, kCT);
                unsigned char* yst = sm + Lay::OFF_Y + s * 16384 + rh * 8192;
                const float* fv = fbuf + (s * 2 + rh) * 64;
#pragma unroll
                for (int c0 = 0; c0 < 32; c0 += 16) {
                    const int tb = wg * 32 + c0;
                    uint32_t v[16];
                    tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + col_y(s) + tb, v);
                    tmem_wait_ld();
                    if (ok) {
#pragma unroll
                        for (int u = 0; u < 16; ++u) {
                            const int t = tb + u;
                            const __nv_bfloat16 yv =
                                __float2bfloat16_rn(__uint_as_float(v[u]) * fv[t]);
                            if (vc == kQ)
                                *reinterpret_cast<__nv_bfloat16*>(yst + sw128_offset(t, rp)) = yv;
                            else if (t < vc)
                                static_cast<__nv_bfloat16*>(a.y)[((tok0 + t) * a.H + h0 + rh) * kP +
                                                                 rp] = yv;
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(&y_free[s]);
                fence_proxy_async();
                named_sync(1, kCT);
                if (ct == 0 && vc == kQ && ok) {
                    tma_store_3d(&map_y, sm + Lay::OFF_Y + s * 16384, 0, h0, (int)tok0);
                    tma_store_3d(&map_y, sm + Lay::OFF_Y + s * 16384 + 8192, 0, h0 + 1, (int)tok0);
                    tma_store_commit();
                }
            }
        }
        if (ct == 0) tma_store_wait_all<0>();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

template <typename K>
cudaError_t set_smem(K kernel, int bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <int N>
cudaError_t forward_n(const Prob& pb, const Args& a, Launch& L) {
    CUtensorMap mx, mb, mc, my;
    if (!make_map(&mx, a.x, pb.T, pb.H, kP) || !make_map(&mb, a.B, pb.T, pb.G, N) ||
        !make_map(&mc, a.C, pb.T, pb.G, N) || !make_map(&my, a.y, pb.T, pb.H, kP))
        return cudaErrorInvalidValue;
    cudaError_t e = launch_seg_table(pb, a, L);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)pb.nseg_max, pb.H / 2);
    const int smem_state = kStateStages * StateSmem::stage_bytes(N) + 2 * kMaxSeg * 4 + 32 +
                           3 * kStateStages * 8 + 8 + 16 + 1024;
    e = set_smem(tc_fwd_state_kernel<N>, smem_state);
    if (e != cudaSuccess) return e;
    L.begin("tc_fwd_state");
    tc_fwd_state_kernel<N><<<grid, kStateThreads, smem_state, L.stream>>>(mx, mb, a);
    e = L.end();
    if (e != cudaSuccess) return e;
    e = launch_state_scan(pb, a, L, a.final_state != nullptr);
    if (e != cudaSuccess) return e;
    e = set_smem(tc_fwd_walk_kernel<N>, WalkLayout<N>::TOTAL);
    if (e != cudaSuccess) return e;
    L.begin("tc_fwd_walk");
    tc_fwd_walk_kernel<N><<<grid, kWalkThreads, WalkLayout<N>::TOTAL, L.stream>>>(mx, mb, mc, my,
                                                                                  a);
    return L.end();
}

}  // namespace

bool tc_supported(int dtype, int P, int N, int Q, int H, int G) {
    return dtype == SSD_DTYPE_BF16 && P == kP && (N == 64 || N == 128) && Q == kQ &&
           ((H / G) % 2) == 0 && encode_fn() != nullptr;
}

cudaError_t tc_forward(const Prob& pb, const Args& a, Launch& L) {
    return pb.N == 128 ? forward_n<128>(pb, a, L) : forward_n<64>(pb, a, L);
}

cudaError_t tc_backward(const Prob& pb, const Args& a, Launch& L) {
    return simt_backward(pb, a, L);
}

}  // namespace ssd
