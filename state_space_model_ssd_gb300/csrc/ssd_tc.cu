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
//     G2  Y[t, (h,p)]    = sum_s L0[t, s] g(s) x_s[(h,p)]            (M=64,  N=128, K=64)
//     G3  Y[t, (h,p)]   += sum_n C_t[n] exp(m) H[(h,p), n]           (M=64,  N=128, K=N)
//         y_t            = f(t) Y[t, .]            = diagonal block + exp(s_t) H C_t
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

#include "simt_body.cuh"
#include "tc_common.cuh"

namespace ssd {

using namespace tc;
using namespace tcc;

namespace {

// ================================================================ SIMT fallback
// Work items (segment, pair of heads) with a chunk whose delta sum exceeds kMaxChunkDecay
// run the SIMT recurrence on the first simt::kSimtThreads threads of the CTA.
template <int N>
__device__ __forceinline__ void fallback_seg_state(const Args& a, int seg, int p, float* sm,
                                                   int bar, int mode) {
    const simt::Ctx cx{(int)threadIdx.x, bar};
    const HeadPair hp = head_pair(a, p);
    for (int hh = 0; hh < (hp.v1 ? 2 : 1); ++hh) {
        if (mode == 0)
            simt::seg_state_body<__nv_bfloat16, kP / 8, N / 32>(a, seg, hp.h0 + hh, sm, cx);
        else
            simt::adj_state_body<__nv_bfloat16, kP / 8, N / 32>(a, seg, hp.h0 + hh, sm, cx);
        cx.sync();
    }
}
template <int N>
__device__ __forceinline__ void fallback_walk(const Args& a, int seg, int p, float* sm, int bar) {
    const simt::Ctx cx{(int)threadIdx.x, bar};
    const HeadPair hp = head_pair(a, p);
    for (int hh = 0; hh < (hp.v1 ? 2 : 1); ++hh) {
        simt::seg_walk_body<__nv_bfloat16, kP / 8, N / 32>(a, seg, hp.h0 + hh, sm, cx);
        cx.sync();
    }
}
template <int N>
__device__ __forceinline__ void fallback_bwd(const Args& a, int seg, int p, float* sm, int bar) {
    const simt::Ctx cx{(int)threadIdx.x, bar};
    const HeadPair hp = head_pair(a, p);
    for (int hh = 0; hh < (hp.v1 ? 2 : 1); ++hh) {
        simt::bwd_walk_body<__nv_bfloat16, kP / 8, N / 32>(a, seg, hp.h0 + hh, sm, cx, true);
        cx.sync();
    }
}

// ================================================================ segment aggregates
// Warps: 0 = TMA producer, 1 = MMA issuer (and TMEM owner), 2..9 = compute.
constexpr int kStateStages = 2;  // with three CTAs per SM (shared memory and TMEM allow it)
constexpr int kStateThreads = 320;  // TMA warp, MMA warp, 8 compute warps
constexpr int kMaxSegChunks = 64;  // chunks per segment the per-chunk scales cover

struct StateSmem {
    // stage = X h0 (8K) | X h1 (8K) | B (N/64 x 8K)
    static constexpr int stage_bytes(int N) { return 16384 + N * 128; }
};

// MODE 0: forward aggregates  A_j  = sum_t exp(Lambda_end - Lambda_t) delta_t x_t B_t^T
//         (operands x, B; also writes the segment log-decay).
// MODE 1: adjoint aggregates Ad_j = sum_u exp(Lambda_u - Lambda_before) dy_u C_u^T
//         (operands dy, C).

template <int N, int MODE>
__global__ void __launch_bounds__(kStateThreads, 3)
    tc_seg_state_kernel(const __grid_constant__ CUtensorMap map_x,
                        const __grid_constant__ CUtensorMap map_b, Args a) {
    if (MODE == 1) {
        // this CTA's share of the fp32 dB / dC accumulators, which the backward walks that
        // follow add into, set to zero
        const long long n4 = a.T * a.G * a.N / 4;
        const long long nb = (long long)gridDim.x * gridDim.y;
        const long long per = (n4 + nb - 1) / nb;
        const long long lo = ((long long)blockIdx.y * gridDim.x + blockIdx.x) * per;
        const long long hi = lo + per < n4 ? lo + per : n4;
        float4* db4 = reinterpret_cast<float4*>(a.dbacc);
        float4* dc4 = reinterpret_cast<float4*>(a.dcacc);
        for (long long i = lo + threadIdx.x; i < hi; i += blockDim.x) {
            db4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            dc4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    // pairs fastest: the CTAs that run together read whole token rows of x (and dy)
    const int seg = blockIdx.x / a.npairs;
    const int pr = blockIdx.x % a.npairs;
    const HeadPair hp = head_pair(a, pr);
    const int h0 = hp.h0;
    if (seg >= a.hdr->nseg) return;
    if (a.fb[(long long)seg * a.npairs + pr]) {
        // a chunk decay beyond the factorisation's range: the SIMT recurrence, both heads
        extern __shared__ float fsm[];
        if (threadIdx.x < simt::kSimtThreads) fallback_seg_state<N>(a, seg, pr, fsm, 3, MODE);
        return;
    }
    const SegInfo si = a.segtab[seg];
    const int g = hp.g;
    const int nchunks = (si.len + kQ - 1) / kQ;
    constexpr int SB = StateSmem::stage_bytes(N);

    extern __shared__ __align__(1024) unsigned char smraw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smraw) + 1023) & ~(uintptr_t)1023);
    unsigned char* stages = sm;
    float* csc = reinterpret_cast<float*>(sm + kStateStages * SB);  // [2 head][kMaxSegChunks]
    float* ctot = csc + 2 * kMaxSegChunks;  // [2 head] first 32 chunks, [2 head] all chunks
    uint64_t* full = reinterpret_cast<uint64_t*>(ctot + 4);
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
            mbar_init(&ready[i], 256);
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
                tma_load_3d(st + 8192, &map_x, &full[s], 0, hp.h1c, tok);
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
        // ---- compute warps: per-token weights from the chunk factor records.  With the
        // records' g(t) = delta_t exp(inc_t - half_c) and f(t) = exp(half_c - inc_t)
        // (inc_t = sum of delta over the chunk up to t, half_c = half the chunk's sum):
        //   MODE 0: w_t = delta_t exp(-(sum of delta over (t, end]))
        //              = g(t) exp(-half_c - 2 sum_{chunks c' > c} half_c'),
        //   MODE 1: w_t = exp(-(sum of delta over [start, t]))
        //              = f(t) exp(-half_c - 2 sum_{chunks c' < c} half_c').
        // The per-chunk scales csc[head][c] come from a scan over the chunks' halves (two
        // warps per head, 32 chunks each); the record values of a chunk are loaded while
        // the chunk before it is scaled.
        const int ct = tid - 64;            // 0..255
        const int cps = a.Ls / kQ;
        const long long slot0 = (long long)seg * cps;
        auto rec = [&](int c, int hh) -> const float* {
            return a.fac + ((slot0 + c) * a.Hf + 2 * pr + hh) * kFacRec;
        };
        float hv = 0.f, pre = 0.f;
        if (ct < 2 * kMaxSegChunks) {
            const int head = ct >> 6, c = ct & 63;
            hv = (c < nchunks) ? rec(c, head)[FAC_HALF] : 0.f;
            pre = warp_scan(hv, lane);  // inclusive, over this warp's 32 chunks
            if (lane == 31 && c < 32) ctot[head] = pre;  // the head's first 32 chunks
        }
        named_sync(2, 256);
        if (ct < 2 * kMaxSegChunks) {
            const int head = ct >> 6, c = ct & 63;
            if (c >= 32) pre += ctot[head];
            if (c == 63) ctot[2 + head] = pre;  // the head's total over all chunks
        }
        named_sync(2, 256);
        if (ct < 2 * kMaxSegChunks) {
            const int head = ct >> 6, c = ct & 63;
            const float tot = ctot[2 + head];
            csc[head * kMaxSegChunks + c] =
                MODE == 0 ? expf(-hv - 2.f * (tot - pre)) : expf(-hv - 2.f * (pre - hv));
            if (MODE == 0 && c == 0 && (head == 0 || hp.v1))
                a.lam[(long long)seg * a.H + h0 + head] = -2.f * tot;
        }
        named_sync(2, 256);  // the scales are visible to all compute warps
        // this thread's 16-byte pieces of the two x tiles: (head slot, row) for i = 0..3
        float wn[4];
        auto load_w = [&](int c) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int idx = ct + 256 * i, hh = idx >> 9, row = (idx & 511) >> 3;
                wn[i] = (c < nchunks && c * kQ + row < si.len)
                            ? __ldg(rec(c, hh) + (MODE == 0 ? FAC_G : FAC_F) + row)
                            : 0.f;
            }
        };
        load_w(0);
        // ---- scale x by the weights in place, chunk by chunk
        for (int c = 0; c < nchunks; ++c) {
            const int s = c % kStateStages;
            float w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) w[i] = wn[i];
            if (c + 1 < nchunks) load_w(c + 1);
            if (!wait_or_abort(&full[s], (c / kStateStages) & 1, abort_flag, a.hdr)) break;
            uint4* xs = reinterpret_cast<uint4*>(stages + s * SB);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int idx = ct + 256 * i;  // 0..1023 16-byte chunks of the two x tiles
                const int hh = idx >> 9;
                xs[idx] = scale_chunk(xs[idx], w[i] * csc[hh * kMaxSegChunks + c]);
            }
            fence_proxy_async();
            mbar_arrive(&ready[s]);
        }
        // ---- epilogue: TMEM -> aggregates A[seg][h] (lane-major: each float4 store of a
        // warp covers 512 contiguous bytes)
        const bool ok = wait_or_abort(done, 0, abort_flag, a.hdr);
        tc_fence_after();
        const int q = warp & 3;
        const int r = 32 * q + lane;  // accumulator row = (head, p)
        const int cbase = (ct >> 7) * (N / 2);  // each of the two warpgroups takes half the columns
        float* Arow = (MODE == 0 ? a.A : a.adj) + ((long long)seg * a.H + h0 + (r >> 6)) * kP * N +
                      lm_row(r & 63, N);
#pragma unroll
        for (int c0 = cbase; c0 < cbase + N / 2; c0 += 16) {
            uint32_t v[16];
            tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + c0, v);
            tmem_wait_ld_regs<16>(v);
            if (ok && ((r >> 6) == 0 || hp.v1)) {  // nothing for a dummy second slot
#pragma unroll
                for (int i = 0; i < 16; i += 4)
                    *reinterpret_cast<float4*>(Arow + (c0 + i) * 32) =
                        make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                                    __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, N);
}

// ================================================================ masked CB^T tiles
// L0[t, s] = (C_t . B_s) [s <= t] for every chunk of every segment and B/C group, as a
// bf16 image of the 128-byte-swizzled K-major operand layout (8 KB: row t at t * 128,
// 16-byte chunk j of it at ((j ^ t) & 7) * 16).  The tile does not depend on the head,
// so it is made once here and copied into each walk's shared memory as it is: the
// forward walk reads it as the A operand of the diagonal block (rows t, K = s), the
// dx/dB walk reads the same bytes as the MN-major A operand of L0^T (rows u, K = t).
// Warps: 0 = TMA producer, 1 = MMA issuer, 2..5 = masking epilogue.  Each CTA takes
// kL0Chunks consecutive chunks of one segment.
// When a.cb32 is set (the backward), the lower triangle of the same products is also
// written in fp32 (kCbTri floats per chunk and group, row t from cb_tri_row(t)): the dC
// walk needs C_t . B_s at the precision its tensor-core products carry it.  write_tile =
// 0 writes only those.
constexpr int kL0Threads = 192;
constexpr int kL0Chunks = 4;

template <int N>
__global__ void __launch_bounds__(kL0Threads)
    tc_l0_kernel(const __grid_constant__ CUtensorMap map_b,
                 const __grid_constant__ CUtensorMap map_c, Args a, int write_tile) {
    const int cps = a.Ls / kQ;                       // chunk slots per segment
    const int parts = (cps + kL0Chunks - 1) / kL0Chunks;
    const int seg = blockIdx.x / parts;
    const int g = blockIdx.y;
    if (seg >= a.hdr->nseg) return;
    const SegInfo si = a.segtab[seg];
    const int c0 = (blockIdx.x % parts) * kL0Chunks;
    const int nloc = min(kL0Chunks, (si.len + kQ - 1) / kQ - c0);
    if (nloc <= 0) return;
    constexpr int STAGE = 2 * N * 128;  // C | B

    extern __shared__ __align__(1024) unsigned char smraw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smraw) + 1023) & ~(uintptr_t)1023);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + 2 * STAGE);
    uint64_t* full = bars + 0;    // [2]
    uint64_t* empty = bars + 2;   // [2]
    uint64_t* tfull = bars + 4;   // [2]
    uint64_t* tfree = bars + 6;   // [2]
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
            mbar_init(&tfull[i], 1);
            mbar_init(&tfree[i], 128);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tslot, 128);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == 0) {
        if (lane == 0) {
            for (int j = 0; j < nloc; ++j) {
                const int s = j & 1;
                if (j >= 2 && !wait_or_abort(&empty[s], ((j >> 1) - 1) & 1, abort_flag, a.hdr))
                    break;
                unsigned char* st = sm + s * STAGE;
                const int tok = (int)(si.start + (long long)(c0 + j) * kQ);
                mbar_expect_tx(&full[s], STAGE);
                for (int nb = 0; nb < N / 64; ++nb) {
                    tma_load_3d(st + nb * 8192, &map_c, &full[s], nb * 64, g, tok);
                    tma_load_3d(st + N * 128 + nb * 8192, &map_b, &full[s], nb * 64, g, tok);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t id = idesc_bf16(64, 64, 0, 0);
            for (int j = 0; j < nloc; ++j) {
                const int s = j & 1, ph = (j >> 1) & 1;
                if (!wait_or_abort(&full[s], ph, abort_flag, a.hdr)) break;
                if (j >= 2 && !wait_or_abort(&tfree[s], ph ^ 1, abort_flag, a.hdr)) break;
                tc_fence_after();
                const uint32_t cs = smem_u32(sm + s * STAGE), bs = cs + N * 128;
#pragma unroll
                for (int k = 0; k < N / 16; ++k) {
                    const uint32_t koff = (k >> 2) * 8192 + (k & 3) * 32;
                    mma_bf16(tmem + s * 64, sw128_desc(cs + koff, 16, 1024),
                             sw128_desc(bs + koff, 16, 1024), id, k > 0 ? 1u : 0u);
                }
                mma_commit(&tfull[s]);
                mma_commit(&empty[s]);
            }
        }
    } else {
        // row tt of the tile; lane half hf holds columns 32 hf .. 32 hf + 31
        const int q = warp & 3;
        const int tt = 16 * q + (lane & 15), hf = lane >> 4;
        const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16);
        for (int j = 0; j < nloc; ++j) {
            const int s = j & 1, ph = (j >> 1) & 1;
            const bool ok = wait_or_abort(&tfull[s], ph, abort_flag, a.hdr);
            tc_fence_after();
            uint32_t v[32];
            tmem_ld16x2<32>(trow + s * 64, &v[0]);
            tmem_ld16x2<32>(trow + s * 64 + 16, &v[16]);
            tmem_wait_ld_regs<32>(v);
            tc_fence_before();
            mbar_arrive(&tfree[s]);
            if (!ok) continue;
            const long long slot = ((long long)seg * cps + c0 + j) * a.G + g;
            unsigned char* tile = a.l0 + slot * 8192 + tt * 128;
            float* crow = a.cb32 ? a.cb32 + slot * kCbTri + cb_tri_row(tt) + 32 * hf : nullptr;
#pragma unroll
            for (int e0 = 0; e0 < 32; e0 += 8) {
                const int e = 32 * hf + e0;
                float f[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) f[u] = (e + u <= tt) ? __uint_as_float(v[e0 + u]) : 0.f;
                if (write_tile)
                    *reinterpret_cast<uint4*>(tile + ((((e >> 3) ^ tt) & 7) << 4)) =
                        make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]),
                                   pack_bf16(f[4], f[5]), pack_bf16(f[6], f[7]));
                if (crow) {
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        if (e + u <= tt) crow[e0 + u] = f[u];
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 128);
}

template <int N>
constexpr int l0_smem_bytes() {
    return 2 * (2 * N * 128) + 8 * 8 + 16 + 1024;
}

// ================================================================ chunk factors
// Per chunk (up to 64 tokens of one segment) and head: delta_t = softplus(raw_t +
// delta_init), the chunk-local log-decay s_t = -sum_{k<=t} delta_k, the reference point
// m = s_end / 2, and f(t) = exp(s_t - m) (zero past the chunk's tokens), g(t) = delta_t
// exp(m - s_t), half = -m.  With them exp(s_t - s_s) = f(t) g(s) / delta_s keeps every
// exponent within |s_end| / 2.  The walks of both passes copy these records instead of
// recomputing them.  One CTA per kFacChunks chunk slots of a segment and group of
// kFacHeads heads: the raw_dt tiles (64 tokens x kFacHeads heads each) are read with
// coalesced loads into shared memory, then one warp scans one (chunk, head)'s 64 tokens,
// two per lane.
constexpr int kFacThreads = 256;
constexpr int kFacHeads = 16;
constexpr int kFacChunks = 4;  // chunks of one segment a CTA takes, all loads in flight at once

__global__ void __launch_bounds__(kFacThreads) tc_factors_kernel(Args a) {
    const int cps = a.Ls / kQ;
    const int groups = (cps + kFacChunks - 1) / kFacChunks;
    const int seg = blockIdx.x / groups, c0 = (blockIdx.x % groups) * kFacChunks;
    if (seg >= a.hdr->nseg) return;
    const SegInfo si = a.segtab[seg];
    const int nch = (si.len + kQ - 1) / kQ;
    if (c0 >= nch) return;
    __shared__ float zt[kFacChunks][kFacHeads][kQ + 1];  // raw_dt + delta_init
    const int ct = threadIdx.x, lane = ct & 31, warp = ct >> 5;
    // record slots hb .. hb + kFacHeads - 1: slot r is lane r % 2 of pair r / 2 (a dummy
    // slot gets an all-zero record)
    const int hb = blockIdx.y * kFacHeads;
    auto head_of = [&](int r) -> int {
        const HeadPair hp = head_pair(a, r >> 1);
        return ((r & 1) == 0 || hp.v1) ? hp.h0 + (r & 1) : -1;
    };
    int hcol[kQ * kFacHeads / kFacThreads];  // the head each of this thread's loads reads
#pragma unroll
    for (int k = 0; k < kQ * kFacHeads / kFacThreads; ++k) {
        const int hh = (ct + kFacThreads * k) % kFacHeads;
        hcol[k] = (hb + hh < a.Hf) ? head_of(hb + hh) : -1;
    }
#pragma unroll
    for (int cc = 0; cc < kFacChunks; ++cc) {
        const int c = c0 + cc;
        const int vc = c < nch ? min(kQ, si.len - c * kQ) : 0;
        const long long tok0 = si.start + (long long)c * kQ;
#pragma unroll
        for (int k = 0; k < kQ * kFacHeads / kFacThreads; ++k) {
            const int idx = ct + kFacThreads * k, t = idx / kFacHeads, hh = idx % kFacHeads;
            float z = 0.f;
            if (t < vc && hcol[k] >= 0) z = a.raw[(tok0 + t) * a.H + hcol[k]] + a.delta_init;
            zt[cc][hh][t] = z;
        }
    }
    __syncthreads();
    // one warp scans one (chunk, head) record's 64 tokens, two per lane
    for (int w = warp; w < kFacChunks * kFacHeads; w += kFacThreads / 32) {
        const int cc = w / kFacHeads, hh = w % kFacHeads;
        const int c = c0 + cc, r = hb + hh;
        if (c >= nch || r >= a.Hf) continue;
        const int vc = min(kQ, si.len - c * kQ), t0 = 2 * lane;
        const bool real = head_of(r) >= 0;
        const float d0 = (real && t0 < vc) ? softplus_f(zt[cc][hh][t0]) : 0.f;
        const float d1 = (real && t0 + 1 < vc) ? softplus_f(zt[cc][hh][t0 + 1]) : 0.f;
        const float incl = warp_scan(d0 + d1, lane);
        float excl = __shfl_up_sync(0xffffffffu, incl, 1);
        if (lane == 0) excl = 0.f;
        const float send = __shfl_sync(0xffffffffu, incl, 31);  // sum of delta over the chunk
        const float half = 0.5f * send;
        const float s0 = excl + d0, s1 = s0 + d1;  // inclusive sums at tokens t0, t0 + 1
        float* rec = a.fac + ((long long)(seg * cps + c) * a.Hf + r) * kFacRec;
        *reinterpret_cast<float2*>(rec + FAC_F + t0) =
            make_float2((real && t0 < vc) ? expf(half - s0) : 0.f,
                        (real && t0 + 1 < vc) ? expf(half - s1) : 0.f);
        *reinterpret_cast<float2*>(rec + FAC_G + t0) =
            make_float2(d0 * expf(s0 - half), d1 * expf(s1 - half));
        *reinterpret_cast<float2*>(rec + FAC_D + t0) = make_float2(d0, d1);
        if (lane < 4) rec[FAC_HALF + lane] = (lane == 0) ? half : 0.f;
        // beyond this decay the factors would leave fp32 range: the (segment, head pair)
        // is evaluated by the SIMT recurrence instead (every writer stores the same 1)
        if (lane == 0 && !(send <= kMaxChunkDecay)) a.fb[(long long)seg * a.npairs + (r >> 1)] = 1;
    }
}

// ================================================================ chunk walk
// x streams from HBM through a ring of kXS slots, refilled kXS - 1 chunks ahead of its
// use (the load latency under full traffic is a few chunk periods); B, C and the L0
// tile, shared by all heads of a group and mostly served by L2, use a ring of two.
// Warps: 0 = TMA producer (x, B, C, the chunk's L0 tile and factor records), 1 = MMA
// issuer of the state chain (G4), 18 = MMA issuer of the y path (G2, G3), 2..17 = four
// compute warpgroups, each with its own task so that the tasks of neighbouring chunks
// overlap:
//   warpgroup 0     x -> g x;
//   warpgroup 1     the y epilogue;
//   warpgroups 2-3  the state update Hs <- gamma (Hs + S) and the G3 operand.
// The groups hand work to each other and to the MMA warp through mbarriers only.
constexpr int kCT = 256;  // compute threads of the backward walks (two warpgroups)
constexpr int kWalkThreads = 64 + 4 * 128 + 32;
constexpr int kFS = 6;    // factor record slots (chunk c uses slot c % kFS)
constexpr int kFSlot = 2 * kFacRec * 4;  // the records of the CTA's two heads
constexpr int kXS = 4;    // x slots (chunk c uses slot c % kXS)

template <int N>
struct WalkLayout {
    static constexpr int XSLOT = 16384;                     // X h0 | X h1
    static constexpr int BCSLOT = 2 * N * 128 + 8192;       // B | C | L0
    static constexpr int C_IN_BC = N * 128;
    static constexpr int L0_IN_BC = 2 * N * 128;
    static constexpr int OFF_X = 0;
    static constexpr int OFF_BC = kXS * XSLOT;
    static constexpr int OFF_H = OFF_BC + 2 * BCSLOT;       // 2 x (N/64) x 16K
    static constexpr int HBUF = (N / 64) * 16384;
    static constexpr int OFF_F = OFF_H + 2 * HBUF;          // factor records [slot][head]
    static constexpr int OFF_BAR = OFF_F + kFS * kFSlot;
    static constexpr int NBAR = 48;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int TOTAL = OFF_MISC + 16 + 1024;  // + alignment slack
};

// TMEM columns: Y (M=64) 2 x 128 | state (M=128) N.  The state lives in TMEM: G4 of
// chunk c adds S_c onto Hs_c there, the state warps turn the sum into Hs_{c+1} in
// place, and G4 of chunk c + 1 waits for that.
__device__ __forceinline__ uint32_t col_y(int b) { return b * 128; }
constexpr uint32_t kColS = 256;

template <int N>
__global__ void __launch_bounds__(kWalkThreads, 1)
    tc_fwd_walk_kernel(const __grid_constant__ CUtensorMap map_x,
                       const __grid_constant__ CUtensorMap map_b,
                       const __grid_constant__ CUtensorMap map_c, Args a) {
    using Lay = WalkLayout<N>;
    // Persistent: the CTA takes items (segment, pair of heads) blockIdx.x, + gridDim.x, ...
    // in segment-major order (neighbouring CTAs share B, C and the L0 tiles in L2).  Every
    // role walks the same items; rings and mbarrier phases run on the CTA's global chunk
    // count gc, so the next item's copies start while the current item's last chunks run.
    const int nseg = a.hdr->nseg;
    const int npairs = a.npairs;
    const int nitems = nseg * npairs;
    if ((int)blockIdx.x >= nitems) return;
    const int cps = a.Ls / kQ;
    struct Item {
        int seg, p, h0, h1c, g, nchunks;
        bool v1;
        SegInfo si;
    };
    auto item_of = [&](int it) -> Item {
        Item r;
        r.seg = it / npairs;
        r.p = it % npairs;
        const HeadPair hp = head_pair(a, r.p);
        r.h0 = hp.h0;
        r.h1c = hp.h1c;
        r.v1 = hp.v1;
        r.g = hp.g;
        r.si = a.segtab[r.seg];
        r.nchunks = (r.si.len + kQ - 1) / kQ;
        return r;
    };

    extern __shared__ __align__(1024) unsigned char smraw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smraw) + 1023) & ~(uintptr_t)1023);
    // factor record of (slot, head): f[64], g[64], delta[64], half
    auto frec = [&](int sl, int head) -> const float* {
        return reinterpret_cast<const float*>(sm + Lay::OFF_F + sl * kFSlot) + head * kFacRec;
    };
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Lay::OFF_BAR);
    uint64_t* full_x = bars + 0;      // [kXS] x of a chunk landed
    uint64_t* empty_x = bars + 4;     // [kXS] x read by the MMAs
    uint64_t* xg_ready = bars + 8;    // [kXS] x scaled in place (warpgroup 0)
    uint64_t* full_bc = bars + 28;    // [2] B, C, L0 of a chunk landed
    uint64_t* empty_bc = bars + 30;   // [2] B, C, L0 read by the MMAs
    uint64_t* s_full = bars + 32;     // S accumulated
    uint64_t* s_free = bars + 33;     // S read by the state warps
    uint64_t* y_full = bars + 12;     // [2] Y accumulated
    uint64_t* y_free = bars + 14;     // [2] Y read by warpgroup 1
    uint64_t* h_ready = bars + 16;    // [2] G3 operand written (state warps)
    uint64_t* h_free = bars + 18;     // [2] G3 operand read by the MMAs
    uint64_t* fac_full = bars + 34;   // [kFS] factor records of a chunk landed
    uint64_t* fac_empty = bars + 40;  // [kFS] factor records of a chunk no longer needed
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + Lay::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int i = 0; i < kXS; ++i) {
            mbar_init(&full_x[i], 1);
            mbar_init(&empty_x[i], 2);  // read by G4 and G2 (two issuing threads)
            mbar_init(&xg_ready[i], 128);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&full_bc[i], 1);
            mbar_init(&empty_bc[i], 2);  // B read by G4, C and L0 by G2 / G3
            mbar_init(&y_full[i], 1);
            mbar_init(&y_free[i], 128);
            mbar_init(&h_ready[i], 256);
            mbar_init(&h_free[i], 1);
        }
        mbar_init(s_full, 1);
        mbar_init(s_free, 256);
        for (int i = 0; i < kFS; ++i) {
            mbar_init(&fac_full[i], 1);
            mbar_init(&fac_empty[i], 128 + 128 + 256);
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
            int gc = 0;
            bool stop = false;
            for (int it = blockIdx.x; it < nitems && !stop; it += gridDim.x) {
                if (a.fb[it]) continue;  // the SIMT recurrence takes it, below
                const Item I = item_of(it);
                for (int c = 0; c < I.nchunks; ++c, ++gc) {
                    const int tok = (int)(I.si.start + (long long)c * kQ);
                    // factor records (slot ring of kFS), x (ring of kXS), B / C / L0 (ring of 2)
                    const int fs = gc % kFS;
                    if (gc >= kFS &&
                        !wait_or_abort(&fac_empty[fs], ((gc / kFS) - 1) & 1, abort_flag, a.hdr)) {
                        stop = true;
                        break;
                    }
                    mbar_expect_tx(&fac_full[fs], kFSlot);
                    bulk_load(sm + Lay::OFF_F + fs * kFSlot,
                              a.fac + ((long long)(I.seg * cps + c) * a.Hf + 2 * I.p) * kFacRec, kFSlot,
                              &fac_full[fs]);
                    const int xs = gc % kXS;
                    if (gc >= kXS &&
                        !wait_or_abort(&empty_x[xs], ((gc / kXS) - 1) & 1, abort_flag, a.hdr)) {
                        stop = true;
                        break;
                    }
                    unsigned char* sx = sm + Lay::OFF_X + xs * Lay::XSLOT;
                    mbar_expect_tx(&full_x[xs], Lay::XSLOT);
                    tma_load_3d(sx, &map_x, &full_x[xs], 0, I.h0, tok);
                    tma_load_3d(sx + 8192, &map_x, &full_x[xs], 0, I.h1c, tok);
                    const int b = gc & 1;
                    if (gc >= 2 &&
                        !wait_or_abort(&empty_bc[b], ((gc >> 1) - 1) & 1, abort_flag, a.hdr)) {
                        stop = true;
                        break;
                    }
                    unsigned char* st = sm + Lay::OFF_BC + b * Lay::BCSLOT;
                    mbar_expect_tx(&full_bc[b], Lay::BCSLOT);
                    for (int nb = 0; nb < N / 64; ++nb) {
                        tma_load_3d(st + nb * 8192, &map_b, &full_bc[b], nb * 64, I.g, tok);
                        tma_load_3d(st + Lay::C_IN_BC + nb * 8192, &map_c, &full_bc[b], nb * 64,
                                    I.g, tok);
                    }
                    bulk_load(st + Lay::L0_IN_BC,
                              a.l0 + (((long long)I.seg * cps + c) * a.G + I.g) * 8192, 8192,
                              &full_bc[b]);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer: state chain
        if (lane == 0) {
            const uint32_t id_s = idesc_bf16(128, N, 1, 1);
            int gc = 0;
            bool stop = false;
            for (int it = blockIdx.x; it < nitems && !stop; it += gridDim.x) {
                if (a.fb[it]) continue;  // the SIMT recurrence takes it, below
                const Item I = item_of(it);
                for (int c = 0; c < I.nchunks; ++c, ++gc) {
                    const int s = gc & 1, ph = (gc >> 1) & 1;
                    const int xsl = gc % kXS, xph = (gc / kXS) & 1;
                    // One s_free and one s_full phase per chunk, also where no G4 is issued
                    // (an item's last chunk), so that this warp and the state warps stay in
                    // step: a parity wait must never be two phases behind its barrier.  The
                    // slot waits keep the "slot read" arrivals below from running ahead.
                    if (!wait_or_abort(&full_bc[s], ph, abort_flag, a.hdr) ||
                        !wait_or_abort(&xg_ready[xsl], xph, abort_flag, a.hdr) ||
                        !wait_or_abort(s_free, gc & 1, abort_flag, a.hdr)) {
                        stop = true;
                        break;
                    }
                    if (c < I.nchunks - 1) {  // G4: Hs_c + S_c in the state columns
                        tc_fence_after();
                        const uint32_t xs = smem_u32(sm + Lay::OFF_X + xsl * Lay::XSLOT);
                        const uint32_t bs = smem_u32(sm + Lay::OFF_BC + s * Lay::BCSLOT);
#pragma unroll
                        for (int k = 0; k < kQ / 16; ++k)
                            mma_bf16(tmem + kColS, sw128_desc(xs + k * 2048, 8192, 1024),
                                     sw128_desc(bs + k * 2048, 8192, 1024), id_s, 1u);
                    }
                    mma_commit(s_full);
                    mma_commit(&empty_x[xsl]);
                    mma_commit(&empty_bc[s]);
                }
            }
        }
    } else if (warp == 18) {
        // ------------------------------------------------ MMA issuer: y path
        if (lane == 0) {
            const uint32_t id_y = idesc_bf16(64, 128, 0, 1);
            const uint32_t id_h = idesc_bf16(64, 128, 0, 0);
            int gc = 0;
            bool stop = false;
            for (int it = blockIdx.x; it < nitems && !stop; it += gridDim.x) {
                if (a.fb[it]) continue;  // the SIMT recurrence takes it, below
                const Item I = item_of(it);
                for (int c = 0; c < I.nchunks; ++c, ++gc) {
                    const int s = gc & 1, ph = (gc >> 1) & 1;
                    const int xsl = gc % kXS, xph = (gc / kXS) & 1;
                    if (!wait_or_abort(&full_bc[s], ph, abort_flag, a.hdr) ||
                        !wait_or_abort(&xg_ready[xsl], xph, abort_flag, a.hdr) ||
                        (gc >= 2 && !wait_or_abort(&y_free[s], ph ^ 1, abort_flag, a.hdr))) {
                        stop = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t xs = smem_u32(sm + Lay::OFF_X + xsl * Lay::XSLOT);
                    const uint32_t bs = smem_u32(sm + Lay::OFF_BC + s * Lay::BCSLOT);
                    const uint32_t cs = bs + Lay::C_IN_BC;
                    const uint32_t l0 = bs + Lay::L0_IN_BC;
                    // G2: diagonal block
#pragma unroll
                    for (int k = 0; k < kQ / 16; ++k)
                        mma_bf16(tmem + col_y(s), sw128_desc(l0 + k * 32, 16, 1024),
                                 sw128_desc(xs + k * 2048, 8192, 1024), id_y, k > 0 ? 1u : 0u);
                    mma_commit(&empty_x[xsl]);
                    // G3: state entering the chunk
                    if (!wait_or_abort(&h_ready[s], ph, abort_flag, a.hdr)) {
                        stop = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t hs = smem_u32(sm + Lay::OFF_H + s * Lay::HBUF);
#pragma unroll
                    for (int k = 0; k < N / 16; ++k) {
                        const uint32_t kc = (k >> 2) * 8192 + (k & 3) * 32;
                        const uint32_t kh = (k >> 2) * 16384 + (k & 3) * 32;
                        mma_bf16(tmem + col_y(s), sw128_desc(cs + kc, 16, 1024),
                                 sw128_desc(hs + kh, 16, 1024), id_h, 1u);
                    }
                    mma_commit(&y_full[s]);
                    mma_commit(&h_free[s]);
                    mma_commit(&empty_bc[s]);
                }
            }
        }
    } else {
        const int ct = tid - 64;        // 0..511
        const int wg = ct >> 7;         // compute warpgroup: task
        const int q = warp & 3;         // TMEM lane quadrant
        const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16);
        if (wg == 0) {
            // ------------------------------------------------ x -> g x
            int gc = 0;
            for (int it = blockIdx.x; it < nitems; it += gridDim.x) {
                if (a.fb[it]) continue;
                const Item I = item_of(it);
                for (int c = 0; c < I.nchunks; ++c, ++gc) {
                    const int xsl = gc % kXS, xph = (gc / kXS) & 1, fs = gc % kFS;
                    bool ok = wait_or_abort(&fac_full[fs], (gc / kFS) & 1, abort_flag, a.hdr);
                    ok = wait_or_abort(&full_x[xsl], xph, abort_flag, a.hdr) && ok;
                    if (ok) {
                        uint4* xs = reinterpret_cast<uint4*>(sm + Lay::OFF_X + xsl * Lay::XSLOT);
                        const float* g0 = frec(fs, 0) + FAC_G;
                        const float* g1 = frec(fs, 1) + FAC_G;
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int idx = ct + 128 * i;  // head = idx / 512, row = (idx / 8) % 64
                            const int row = (idx >> 3) & 63;
                            xs[idx] = scale_chunk(xs[idx], (idx >> 9) ? g1[row] : g0[row]);
                        }
                    }
                    fence_proxy_async();
                    mbar_arrive(&xg_ready[xsl]);
                    mbar_arrive(&fac_empty[fs]);
                }
            }
        } else if (wg == 1) {
            // ------------------------------------------------ the y epilogue
            const int tt = 16 * q + (lane & 15);  // M=64 accumulator row (token)
            const int hf = lane >> 4;             // M=64 column half of this lane
            int gc = 0;
            for (int it = blockIdx.x; it < nitems; it += gridDim.x) {
                if (a.fb[it]) continue;
                const Item I = item_of(it);
                for (int c = 0; c < I.nchunks; ++c, ++gc) {
                    // y of the chunk: lane half hf holds head hf, p = 0..63 of token tt
                    const int s = gc & 1, ph = (gc >> 1) & 1, sl = gc % kFS;
                    const int vc = min(kQ, I.si.len - c * kQ);
                    const long long tok0 = I.si.start + (long long)c * kQ;
                    bool ok = wait_or_abort(&fac_full[sl], (gc / kFS) & 1, abort_flag, a.hdr);
                    ok = wait_or_abort(&y_full[s], ph, abort_flag, a.hdr) && ok;
                    tc_fence_after();
                    const float fv = frec(sl, hf)[FAC_F + tt];
                    mbar_arrive(&fac_empty[sl]);
                    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.y) +
                                                          ((tok0 + tt) * a.H + I.h0 + hf) * kP);
                    const bool wide = (reinterpret_cast<uintptr_t>(a.y) & 31) == 0;
#pragma unroll
                    for (int j = 0; j < 64; j += 32) {
                        uint32_t v[32];
                        tmem_ld16x2<64>(trow + col_y(s) + j, &v[0]);
                        tmem_ld16x2<64>(trow + col_y(s) + j + 16, &v[16]);
                        tmem_wait_ld_regs<32>(v);
                        if (j == 32) {
                            tc_fence_before();
                            mbar_arrive(&y_free[s]);
                        }
                        if (ok && tt < vc && (hf == 0 || I.v1)) {
                            store_bf16x16(dst + (j >> 3), v, fv, wide);
                            store_bf16x16(dst + ((j + 16) >> 3), v + 16, fv, wide);
                        }
                    }
                }
            }
        } else {
            // ------------------------------------------------ state chain
            // The state is kept pre-scaled for its next chunk, Hs_c = exp(m_c) H_c, in the
            // TMEM state columns (row r = (head, p), columns [n0, n0 + N / 2) per
            // warpgroup).  G4 leaves Hs_c + S_c there; this group rewrites it as
            //   Hs_{c+1} = exp(m_{c+1} + s_end_c / 2) (Hs_c + S_c)      (m_c = s_end_c / 2)
            // and stores bf16(Hs_{c+1}), the G3 operand of the next chunk.
            constexpr int NH = N / 2;
            const int r = 32 * q + lane;
            const int rh = r >> 6, rp = r & 63;
            const int n0 = (wg - 2) * NH;
            const uint32_t tcol = trow + kColS + n0;
            // bf16 of 32 state values (columns n0 + c0 ..) into the G3 operand of chunk gcc
            auto write_h32 = [&](int gcc, int c0, const float* h) {
                unsigned char* hb = sm + Lay::OFF_H + (gcc & 1) * Lay::HBUF + r * 128;
#pragma unroll
                for (int c8 = 0; c8 < 32; c8 += 8) {
                    const int n = n0 + c0 + c8;
                    const uint4 v = make_uint4(pack_bf16(h[c8], h[c8 + 1]),
                                               pack_bf16(h[c8 + 2], h[c8 + 3]),
                                               pack_bf16(h[c8 + 4], h[c8 + 5]),
                                               pack_bf16(h[c8 + 6], h[c8 + 7]));
                    *reinterpret_cast<uint4*>(hb + (n >> 6) * 16384 +
                                              (((((n & 63) >> 3) ^ r) & 7) << 4)) = v;
                }
            };
            int gc = 0;
            for (int it = blockIdx.x; it < nitems; it += gridDim.x) {
                if (a.fb[it]) continue;
                const Item I = item_of(it);
                {
                    // the item's first chunk: state entering the segment; its G3 operand
                    // buffer was last read by G3 of global chunk gc - 2
                    wait_or_abort(&fac_full[gc % kFS], (gc / kFS) & 1, abort_flag, a.hdr);
                    if (gc >= 2)
                        wait_or_abort(&h_free[gc & 1], ((gc - 2) >> 1) & 1, abort_flag, a.hdr);
                    // exp(m_0); a dummy second slot starts (and stays) at zero
                    const float sc0 = (rh == 0 || I.v1) ? expf(-frec(gc % kFS, rh)[FAC_HALF]) : 0.f;
                    const float* Hin =
                        a.A + ((long long)I.seg * a.H + I.h0 + (I.v1 ? rh : 0)) * kP * N +
                        lm_row(rp, N) + n0 * 32;
#pragma unroll
                    for (int c0 = 0; c0 < NH; c0 += 32) {
                        float h[32];
#pragma unroll
                        for (int i = 0; i < 32; i += 4) {
                            const float4 v = *reinterpret_cast<const float4*>(Hin + (c0 + i) * 32);
                            h[i] = v.x * sc0;
                            h[i + 1] = v.y * sc0;
                            h[i + 2] = v.z * sc0;
                            h[i + 3] = v.w * sc0;
                        }
                        tmem_st16(tcol + c0, reinterpret_cast<const uint32_t*>(&h[0]));
                        tmem_st16(tcol + c0 + 16, reinterpret_cast<const uint32_t*>(&h[16]));
                        write_h32(gc, c0, h);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(s_free);
                    fence_proxy_async();
                    mbar_arrive(&h_ready[gc & 1]);
                }
                for (int c = 0; c + 1 < I.nchunks; ++c, ++gc) {
                    const int sl = gc % kFS, sn = (gc + 1) % kFS;
                    bool ok = wait_or_abort(&fac_full[sn], ((gc + 1) / kFS) & 1, abort_flag, a.hdr);
                    const float gam = expf(-(frec(sl, rh)[FAC_HALF] + frec(sn, rh)[FAC_HALF]));
                    // the G3 operand buffer of chunk gc + 1 was last read by G3 of gc - 1
                    if (gc >= 1)
                        wait_or_abort(&h_free[(gc + 1) & 1], ((gc - 1) >> 1) & 1, abort_flag,
                                      a.hdr);
                    ok = wait_or_abort(s_full, gc & 1, abort_flag, a.hdr) && ok;
                    tc_fence_after();
#pragma unroll
                    for (int c0 = 0; c0 < NH; c0 += 32) {
                        uint32_t v[32];
                        tmem_ld16(tcol + c0, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
                        tmem_ld16(tcol + c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
                        tmem_wait_ld_regs<32>(v);
                        float h[32];
#pragma unroll
                        for (int u = 0; u < 32; ++u) h[u] = ok ? gam * __uint_as_float(v[u]) : 0.f;
                        tmem_st16(tcol + c0, reinterpret_cast<const uint32_t*>(&h[0]));
                        tmem_st16(tcol + c0 + 16, reinterpret_cast<const uint32_t*>(&h[16]));
                        write_h32(gc + 1, c0, h);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(s_free);
                    mbar_arrive(&fac_empty[sl]);
                    fence_proxy_async();
                    mbar_arrive(&h_ready[(gc + 1) & 1]);
                }
                // the item's last chunk: no update, but its s_full phase is consumed
                wait_or_abort(s_full, gc & 1, abort_flag, a.hdr);
                mbar_arrive(&fac_empty[gc % kFS]);
                ++gc;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------- the walk at two CTAs an SM
// N = 64 (the long-sequence workload): the same chunk walk with one Y accumulator, one G3
// operand buffer, two x slots, four factor record slots and 11 warps, so that two CTAs
// share each SM (103 KB of shared memory, 256 TMEM columns and 352 threads each) and
// each hides the other's hand-off latency.  Warps: 0 = TMA producer, 1 = MMA issuer of
// G4 (onto the state in TMEM), 10 = MMA issuer of G2 and G3, 2..5 = x -> g x of a chunk,
// then the y epilogue of the chunk before it, 6..9 = the state update and the G3 operand.
constexpr int kWalk2Threads = 64 + 2 * 128 + 32;
constexpr int kW2XS = 2;  // x slots
constexpr int kW2FS = 4;  // factor record slots

struct Walk2Layout {
    static constexpr int XSLOT = 16384;               // X h0 | X h1
    static constexpr int BCSLOT = 2 * 64 * 128 + 8192;  // B | C | L0
    static constexpr int C_IN_BC = 64 * 128;
    static constexpr int L0_IN_BC = 2 * 64 * 128;
    static constexpr int OFF_X = 0;
    static constexpr int OFF_BC = kW2XS * XSLOT;
    static constexpr int OFF_H = OFF_BC + 2 * BCSLOT;   // 16 KB
    static constexpr int OFF_F = OFF_H + 16384;
    static constexpr int OFF_BAR = OFF_F + kW2FS * kFSlot;
    static constexpr int NBAR = 24;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int TOTAL = OFF_MISC + 16 + 1024;
};
static_assert(2 * (Walk2Layout::TOTAL + 1024) <= 233472, "two walk CTAs an SM");

__global__ void __launch_bounds__(kWalk2Threads, 2)
    tc_fwd_walk2_kernel(const __grid_constant__ CUtensorMap map_x,
                        const __grid_constant__ CUtensorMap map_b,
                        const __grid_constant__ CUtensorMap map_c, Args a) {
    constexpr int N = 64;
    using Lay = Walk2Layout;
    const int nseg = a.hdr->nseg;
    const int npairs = a.npairs;
    const int nitems = nseg * npairs;
    if ((int)blockIdx.x >= nitems) return;
    const int cps = a.Ls / kQ;
    struct Item {
        int seg, p, h0, h1c, g, nchunks;
        bool v1;
        SegInfo si;
    };
    auto item_of = [&](int it) -> Item {
        Item r;
        r.seg = it / npairs;
        r.p = it % npairs;
        const HeadPair hp = head_pair(a, r.p);
        r.h0 = hp.h0;
        r.h1c = hp.h1c;
        r.v1 = hp.v1;
        r.g = hp.g;
        r.si = a.segtab[r.seg];
        r.nchunks = (r.si.len + kQ - 1) / kQ;
        return r;
    };

    extern __shared__ __align__(1024) unsigned char smraw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smraw) + 1023) & ~(uintptr_t)1023);
    auto frec = [&](int sl, int head) -> const float* {
        return reinterpret_cast<const float*>(sm + Lay::OFF_F + sl * kFSlot) + head * kFacRec;
    };
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Lay::OFF_BAR);
    uint64_t* full_x = bars + 0;      // [2] x of a chunk landed
    uint64_t* empty_x = bars + 2;     // [2] x read by G4 and G2
    uint64_t* xg_ready = bars + 4;    // [2] x scaled in place
    uint64_t* full_bc = bars + 6;     // [2] B, C, L0 landed
    uint64_t* empty_bc = bars + 8;    // [2] B, C, L0 read by the MMAs
    uint64_t* y_full = bars + 10;     // Y accumulated
    uint64_t* y_free = bars + 11;     // Y read by the epilogue
    uint64_t* h_ready = bars + 12;    // G3 operand written
    uint64_t* h_free = bars + 13;     // G3 operand read by the MMAs
    uint64_t* s_full = bars + 14;     // S accumulated onto the state
    uint64_t* s_free = bars + 15;     // the state rescaled in place
    uint64_t* fac_full = bars + 16;   // [kW2FS]
    uint64_t* fac_empty = bars + 20;  // [kW2FS]
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + Lay::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
    constexpr uint32_t kColY = 0, kColSt = 128;  // TMEM: Y (M=64) 128 columns | state N

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int i = 0; i < kW2XS; ++i) {
            mbar_init(&full_x[i], 1);
            mbar_init(&empty_x[i], 2);
            mbar_init(&xg_ready[i], 128);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&full_bc[i], 1);
            mbar_init(&empty_bc[i], 2);
        }
        mbar_init(y_full, 1);
        mbar_init(y_free, 128);
        mbar_init(h_ready, 128);
        mbar_init(h_free, 1);
        mbar_init(s_full, 1);
        mbar_init(s_free, 128);
        for (int i = 0; i < kW2FS; ++i) {
            mbar_init(&fac_full[i], 1);
            mbar_init(&fac_empty[i], 128 + 128 + 128);  // scaling, epilogue, state
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tslot, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int gc = 0;
            bool stop = false;
            for (int it = blockIdx.x; it < nitems && !stop; it += gridDim.x) {
                if (a.fb[it]) continue;
                const Item I = item_of(it);
                for (int c = 0; c < I.nchunks; ++c, ++gc) {
                    const int tok = (int)(I.si.start + (long long)c * kQ);
                    const int fs = gc % kW2FS;
                    if (gc >= kW2FS &&
                        !wait_or_abort(&fac_empty[fs], ((gc / kW2FS) - 1) & 1, abort_flag, a.hdr)) {
                        stop = true;
                        break;
                    }
                    mbar_expect_tx(&fac_full[fs], kFSlot);
                    bulk_load(sm + Lay::OFF_F + fs * kFSlot,
                              a.fac + ((long long)(I.seg * cps + c) * a.Hf + 2 * I.p) * kFacRec, kFSlot,
                              &fac_full[fs]);
                    const int xs = gc % kW2XS;
                    if (gc >= kW2XS &&
                        !wait_or_abort(&empty_x[xs], ((gc / kW2XS) - 1) & 1, abort_flag, a.hdr)) {
                        stop = true;
                        break;
                    }
                    unsigned char* sx = sm + Lay::OFF_X + xs * Lay::XSLOT;
                    mbar_expect_tx(&full_x[xs], Lay::XSLOT);
                    tma_load_3d(sx, &map_x, &full_x[xs], 0, I.h0, tok);
                    tma_load_3d(sx + 8192, &map_x, &full_x[xs], 0, I.h1c, tok);
                    const int b = gc & 1;
                    if (gc >= 2 &&
                        !wait_or_abort(&empty_bc[b], ((gc >> 1) - 1) & 1, abort_flag, a.hdr)) {
                        stop = true;
                        break;
                    }
                    unsigned char* st = sm + Lay::OFF_BC + b * Lay::BCSLOT;
                    mbar_expect_tx(&full_bc[b], Lay::BCSLOT);
                    tma_load_3d(st, &map_b, &full_bc[b], 0, I.g, tok);
                    tma_load_3d(st + Lay::C_IN_BC, &map_c, &full_bc[b], 0, I.g, tok);
                    bulk_load(st + Lay::L0_IN_BC,
                              a.l0 + (((long long)I.seg * cps + c) * a.G + I.g) * 8192, 8192,
                              &full_bc[b]);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer: G4 onto the state
        if (lane == 0) {
            const uint32_t id_s = idesc_bf16(128, N, 1, 1);
            int gc = 0;
            bool stop = false;
            for (int it = blockIdx.x; it < nitems && !stop; it += gridDim.x) {
                if (a.fb[it]) continue;
                const Item I = item_of(it);
                for (int c = 0; c < I.nchunks; ++c, ++gc) {
                    const int b = gc & 1, bph = (gc >> 1) & 1;
                    const int xsl = gc % kW2XS, xph = (gc / kW2XS) & 1;
                    // one s_free and one s_full phase per chunk, also where no G4 is issued
                    if (!wait_or_abort(&full_bc[b], bph, abort_flag, a.hdr) ||
                        !wait_or_abort(&xg_ready[xsl], xph, abort_flag, a.hdr) ||
                        !wait_or_abort(s_free, gc & 1, abort_flag, a.hdr)) {
                        stop = true;
                        break;
                    }
                    if (c < I.nchunks - 1) {
                        tc_fence_after();
                        const uint32_t xs = smem_u32(sm + Lay::OFF_X + xsl * Lay::XSLOT);
                        const uint32_t bs = smem_u32(sm + Lay::OFF_BC + b * Lay::BCSLOT);
#pragma unroll
                        for (int k = 0; k < kQ / 16; ++k)
                            mma_bf16(tmem + kColSt, sw128_desc(xs + k * 2048, 8192, 1024),
                                     sw128_desc(bs + k * 2048, 8192, 1024), id_s, 1u);
                    }
                    mma_commit(s_full);
                    mma_commit(&empty_x[xsl]);
                    mma_commit(&empty_bc[b]);
                }
            }
        }
    } else if (warp == 10) {
        // ------------------------------------------------ MMA issuer: G2, G3 into Y
        if (lane == 0) {
            const uint32_t id_y = idesc_bf16(64, 128, 0, 1);
            const uint32_t id_h = idesc_bf16(64, 128, 0, 0);
            int gc = 0;
            bool stop = false;
            for (int it = blockIdx.x; it < nitems && !stop; it += gridDim.x) {
                if (a.fb[it]) continue;
                const Item I = item_of(it);
                for (int c = 0; c < I.nchunks; ++c, ++gc) {
                    const int b = gc & 1, bph = (gc >> 1) & 1;
                    const int xsl = gc % kW2XS, xph = (gc / kW2XS) & 1;
                    if (!wait_or_abort(&full_bc[b], bph, abort_flag, a.hdr) ||
                        !wait_or_abort(&xg_ready[xsl], xph, abort_flag, a.hdr) ||
                        (gc >= 1 && !wait_or_abort(y_free, (gc - 1) & 1, abort_flag, a.hdr))) {
                        stop = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t xs = smem_u32(sm + Lay::OFF_X + xsl * Lay::XSLOT);
                    const uint32_t bs = smem_u32(sm + Lay::OFF_BC + b * Lay::BCSLOT);
                    const uint32_t cs = bs + Lay::C_IN_BC;
                    const uint32_t l0 = bs + Lay::L0_IN_BC;
#pragma unroll
                    for (int k = 0; k < kQ / 16; ++k)
                        mma_bf16(tmem + kColY, sw128_desc(l0 + k * 32, 16, 1024),
                                 sw128_desc(xs + k * 2048, 8192, 1024), id_y, k > 0 ? 1u : 0u);
                    mma_commit(&empty_x[xsl]);
                    if (!wait_or_abort(h_ready, gc & 1, abort_flag, a.hdr)) {
                        stop = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t hs = smem_u32(sm + Lay::OFF_H);
#pragma unroll
                    for (int k = 0; k < N / 16; ++k)
                        mma_bf16(tmem + kColY, sw128_desc(cs + k * 32, 16, 1024),
                                 sw128_desc(hs + k * 32, 16, 1024), id_h, 1u);
                    mma_commit(y_full);
                    mma_commit(h_free);
                    mma_commit(&empty_bc[b]);
                }
            }
        }
    } else if (warp >= 2 && warp < 10) {
        const int ct = tid - 64;        // 0..255
        const int wg = ct >> 7;
        const int q = warp & 3;
        const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16);
        if (wg == 0) {
            // ------------------------------------------------ x -> g x, the y epilogue
            const int tt = 16 * q + (lane & 15);
            const int hf = lane >> 4;
            const bool wide = (reinterpret_cast<uintptr_t>(a.y) & 31) == 0;
            auto scale_x = [&](int gcs) {
                const int xsl = gcs % kW2XS, xph = (gcs / kW2XS) & 1, fs = gcs % kW2FS;
                bool ok = wait_or_abort(&fac_full[fs], (gcs / kW2FS) & 1, abort_flag, a.hdr);
                ok = wait_or_abort(&full_x[xsl], xph, abort_flag, a.hdr) && ok;
                if (ok) {
                    uint4* xs = reinterpret_cast<uint4*>(sm + Lay::OFF_X + xsl * Lay::XSLOT);
#pragma unroll
                    for (int i0 = 0; i0 < 8; i0 += 4) {
                        uint4 v[4];
                        float gv[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int idx = ct + 128 * (i0 + i);  // head idx / 512, row (idx / 8) % 64
                            v[i] = xs[idx];
                            gv[i] = frec(fs, idx >> 9)[FAC_G + ((idx >> 3) & 63)];
                        }
#pragma unroll
                        for (int i = 0; i < 4; ++i) xs[ct + 128 * (i0 + i)] = scale_chunk(v[i], gv[i]);
                    }
                }
                fence_proxy_async();
                mbar_arrive(&xg_ready[xsl]);
                mbar_arrive(&fac_empty[fs]);
            };
            struct YChunk {
                long long tok0;
                int vc, h0;
                bool v1;
            };
            auto drain_y = [&](int gce, const YChunk& Y) {
                const int sl = gce % kW2FS;
                bool ok = wait_or_abort(&fac_full[sl], (gce / kW2FS) & 1, abort_flag, a.hdr);
                ok = wait_or_abort(y_full, gce & 1, abort_flag, a.hdr) && ok;
                tc_fence_after();
                const float fv = frec(sl, hf)[FAC_F + tt];
                mbar_arrive(&fac_empty[sl]);
                uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.y) +
                                                      ((Y.tok0 + tt) * a.H + Y.h0 + hf) * kP);
#pragma unroll
                for (int j = 0; j < 64; j += 32) {
                    uint32_t v[32];
                    tmem_ld16x2<64>(trow + kColY + j, &v[0]);
                    tmem_ld16x2<64>(trow + kColY + j + 16, &v[16]);
                    tmem_wait_ld_regs<32>(v);
                    if (j == 32) {
                        tc_fence_before();
                        mbar_arrive(y_free);
                    }
                    if (ok && tt < Y.vc && (hf == 0 || Y.v1)) {
                        store_bf16x16(dst + (j >> 3), v, fv, wide);
                        store_bf16x16(dst + ((j + 16) >> 3), v + 16, fv, wide);
                    }
                }
            };
            int gc = 0;
            YChunk prev = {0, 0, 0, false};
            for (int it = blockIdx.x; it < nitems; it += gridDim.x) {
                if (a.fb[it]) continue;
                const Item I = item_of(it);
                for (int c = 0; c < I.nchunks; ++c, ++gc) {
                    scale_x(gc);
                    if (gc >= 1) drain_y(gc - 1, prev);
                    prev.tok0 = I.si.start + (long long)c * kQ;
                    prev.vc = min(kQ, I.si.len - c * kQ);
                    prev.h0 = I.h0;
                    prev.v1 = I.v1;
                }
            }
            if (gc >= 1) drain_y(gc - 1, prev);
        } else {
            // ------------------------------------------------ state chain
            // as in the one-CTA walk: the state Hs_c stays in TMEM, G4 adds S_c onto it, and
            // this group rewrites it as Hs_{c+1} = gamma (Hs_c + S_c) and stores bf16(Hs_{c+1}),
            // the G3 operand (row r = (head, p), all N columns)
            const int r = 32 * q + lane;
            const int rh = r >> 6, rp = r & 63;
            const uint32_t tcol = trow + kColSt;
            auto write_h32 = [&](int c0, const float* h) {
                unsigned char* hb = sm + Lay::OFF_H + r * 128;
#pragma unroll
                for (int c8 = 0; c8 < 32; c8 += 8) {
                    const int n = c0 + c8;
                    const uint4 v = make_uint4(pack_bf16(h[c8], h[c8 + 1]),
                                               pack_bf16(h[c8 + 2], h[c8 + 3]),
                                               pack_bf16(h[c8 + 4], h[c8 + 5]),
                                               pack_bf16(h[c8 + 6], h[c8 + 7]));
                    *reinterpret_cast<uint4*>(hb + ((((n >> 3) ^ r) & 7) << 4)) = v;
                }
            };
            int gc = 0;
            for (int it = blockIdx.x; it < nitems; it += gridDim.x) {
                if (a.fb[it]) continue;
                const Item I = item_of(it);
                {
                    // the item's first chunk: state entering the segment; the G3 operand
                    // buffer was last read by G3 of global chunk gc - 1
                    wait_or_abort(&fac_full[gc % kW2FS], (gc / kW2FS) & 1, abort_flag, a.hdr);
                    if (gc >= 1) wait_or_abort(h_free, (gc - 1) & 1, abort_flag, a.hdr);
                    const float sc0 = (rh == 0 || I.v1) ? expf(-frec(gc % kW2FS, rh)[FAC_HALF]) : 0.f;
                    const float* Hin =
                        a.A + ((long long)I.seg * a.H + I.h0 + (I.v1 ? rh : 0)) * kP * N +
                        lm_row(rp, N);
#pragma unroll
                    for (int c0 = 0; c0 < N; c0 += 32) {
                        float h[32];
#pragma unroll
                        for (int i = 0; i < 32; i += 4) {
                            const float4 v = *reinterpret_cast<const float4*>(Hin + (c0 + i) * 32);
                            h[i] = v.x * sc0;
                            h[i + 1] = v.y * sc0;
                            h[i + 2] = v.z * sc0;
                            h[i + 3] = v.w * sc0;
                        }
                        tmem_st16(tcol + c0, reinterpret_cast<const uint32_t*>(&h[0]));
                        tmem_st16(tcol + c0 + 16, reinterpret_cast<const uint32_t*>(&h[16]));
                        write_h32(c0, h);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(s_free);
                    fence_proxy_async();
                    mbar_arrive(h_ready);
                }
                for (int c = 0; c + 1 < I.nchunks; ++c, ++gc) {
                    const int sl = gc % kW2FS, sn = (gc + 1) % kW2FS;
                    bool ok = wait_or_abort(&fac_full[sn], ((gc + 1) / kW2FS) & 1, abort_flag, a.hdr);
                    const float gam = expf(-(frec(sl, rh)[FAC_HALF] + frec(sn, rh)[FAC_HALF]));
                    // the G3 operand buffer is rewritten once G3 of this chunk has read it
                    wait_or_abort(h_free, gc & 1, abort_flag, a.hdr);
                    ok = wait_or_abort(s_full, gc & 1, abort_flag, a.hdr) && ok;
                    tc_fence_after();
#pragma unroll
                    for (int c0 = 0; c0 < N; c0 += 32) {
                        uint32_t v[32];
                        tmem_ld16(tcol + c0, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
                        tmem_ld16(tcol + c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
                        tmem_wait_ld_regs<32>(v);
                        float h[32];
#pragma unroll
                        for (int u = 0; u < 32; ++u) h[u] = ok ? gam * __uint_as_float(v[u]) : 0.f;
                        tmem_st16(tcol + c0, reinterpret_cast<const uint32_t*>(&h[0]));
                        tmem_st16(tcol + c0 + 16, reinterpret_cast<const uint32_t*>(&h[16]));
                        write_h32(c0, h);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(s_free);
                    mbar_arrive(&fac_empty[sl]);
                    fence_proxy_async();
                    mbar_arrive(h_ready);
                }
                // the item's last chunk: no update, but its s_full phase is consumed
                wait_or_abort(s_full, gc & 1, abort_flag, a.hdr);
                mbar_arrive(&fac_empty[gc % kW2FS]);
                ++gc;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 256);
}

// The forward walk of the items (segment, pair of heads) whose chunk decays leave the
// factorisation's range (tc_fwd_walk skips them): the SIMT recurrence, a persistent grid
// over the items; it exits at once when there are none.
template <int N>
__global__ void __launch_bounds__(simt::kSimtThreads) tc_fallback_walk_kernel(Args a) {
    extern __shared__ float fsm[];
    const int npairs = a.npairs;
    const int nitems = a.hdr->nseg * npairs;
    for (int it = blockIdx.x; it < nitems; it += gridDim.x)
        if (a.fb[it]) fallback_walk<N>(a, it / npairs, it % npairs, fsm, 1);
}

// ================================================================ backward walks
// Both backward kernels walk a segment chunk by chunk for one pair of heads,
// with the same warp roles as the forward walk (0 = TMA, 1 = MMA, 2..9 =
// compute).  Per chunk: f(t) = exp(s_t - m), g(t) = delta_t exp(m - s_t) as in
// the forward; xg = g x (both walks) and dyf = f dy (dx/dB walk) are scaled in place
// in the stage.
//
// tc_bwd_dc (chunks in order, state Hs_c = exp(m_c) H_c as in the forward walk):
//   P1_h[t, s] = dyf_t . xg_s                                  (M=64, N=64, K=P)
//   W_h        = P1_h masked to s <= t                           (epilogue, bf16)
//   dC_h[t, .] = W_h B + dyf_h Hs_h   = H_t^T dy_t for head h    (M=64, N=N, K=64 + 64)
//   r_t,h      = C_t . dC_h[t, .]     = dy_t . y_t
//   dC         = sum over the pair, added into the fp32 accumulator
// tc_bwd_dxdb (chunks in reverse, adjoint Gs_c = exp(s_end - m) G_c where G_c
// arrives at the chunk end from later tokens; Gs_{c-1} = gamma (Gs_c + S'_c)):
//   S'[(h,p), n] = sum_u dyf_u[(h,p)] C_u[n]                     (M=128, N=N, K=64)
//   L0T[t, u]    = (B_t . C_u) [u >= t]                          (M=64, N=64, K=N)
//   DX[t,(h,p)]  = sum_u L0T[t,u] dyf_u[(h,p)] + B_t . Gs[(h,p)]   (M=64, N=128)
//   dx_t         = g(t) DX[t, .],  q_t = x_t . dx_t
//   P2_h[t, u]   = xg_t . dyf_u masked to u >= t                 (M=64, N=64, K=P)
//   dB[t, .]     = sum_h P2_h C + xg_h Gs_h                      (M=64, N=N)
//   d_raw_t = sigmoid(z_t) (q_t / delta_t - sum_{u >= t in the segment} (r_u - q_u) - <G_seg, H_end>)
constexpr int kBwdThreads = 320;

template <int N>
struct BwdLayout {
    static constexpr int STAGE = 32768 + 2 * N * 128;      // x h0|h1, dy h0|h1, B, C
    static constexpr int OFF_STAGE = 0;
    static constexpr int OFF_T0 = 2 * STAGE;               // two 8K operand tiles (W / P2m)
    static constexpr int OFF_S = OFF_T0 + 16384;           // state operand, 2 x (N/64) x 16K
    static constexpr int SBUF = (N / 64) * 16384;
    static constexpr int OFF_CB = OFF_S + 2 * SBUF;        // fp32 C B^T triangle of a chunk
    static constexpr int OFF_F = OFF_CB + kCbTri * 4;      // f, g, delta: [2 buf][2 head][64] each
    static constexpr int OFF_SC = OFF_F + 3 * 2 * 2 * 64 * 4;  // half: [2 buf][2 head][4]
    static constexpr int OFF_RQ = OFF_SC + 2 * 2 * 4 * 4;      // [2 wg][2 head][64]
    static constexpr int OFF_RED = OFF_RQ + 2 * 2 * 64 * 4;    // [16]
    static constexpr int OFF_RI = OFF_RED + 64;                // [2 head][64]
    static constexpr int OFF_BAR = OFF_RI + 2 * 64 * 4;
    static constexpr int NBAR = 16;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int TOTAL = OFF_MISC + 16 + 1024;
};

__device__ __forceinline__ uint64_t kdesc(uint32_t base, int k16, uint32_t kblock) {
    return sw128_desc(base + (k16 >> 2) * kblock + (k16 & 3) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t mdesc(uint32_t base, int k16, uint32_t lbo) {
    return sw128_desc(base + k16 * 2048, lbo, 1024);
}

// Per-chunk factors of the dC walk, two chunk buffers (copied from the records).
struct ChunkFactors {
    float* fbuf;  // [2][2][64]
    float* gbuf;
    float* dbuf;
    float* scal;  // [2][2][4]: half
    float* red;
};

// Thread ct < 128's values (head ct / 64, token ct % 64) of chunk cc's factor records,
// loaded early so that the copy into shared memory does not wait for memory.
struct FacVals {
    float f, g, d, half;
};
__device__ __forceinline__ FacVals load_fac_vals(const Args& a, int seg, int pr, int cc,
                                                 int nchunks, int ct) {
    FacVals v = {0.f, 0.f, 0.f, 0.f};
    if (ct < 128 && cc >= 0 && cc < nchunks) {
        const int head = ct >> 6, t = ct & 63;
        const float* rec =
            a.fac + ((long long)(seg * (a.Ls / kQ) + cc) * a.Hf + 2 * pr + head) * kFacRec;
        v.f = rec[FAC_F + t];
        v.g = rec[FAC_G + t];
        v.d = rec[FAC_D + t];
        v.half = rec[FAC_HALF];
    }
    return v;
}
// Stores chunk cc's factors into buffer cc & 1 (all kCT compute threads must call).
__device__ __forceinline__ void bwd_factors(const ChunkFactors& F, const FacVals& v, int cc,
                                            int ct) {
    named_sync(1, kCT);
    if (ct < 128) {
        const int head = ct >> 6, t = ct & 63, b = cc & 1;
        F.fbuf[(b * 2 + head) * 64 + t] = v.f;
        F.gbuf[(b * 2 + head) * 64 + t] = v.g;
        F.dbuf[(b * 2 + head) * 64 + t] = v.d;
        if (t == 0) F.scal[(b * 2 + head) * 4 + 0] = v.half;
    }
    named_sync(1, kCT);
}

// x -> g x and dy -> f dy in place (the 2 x tiles and the 2 dy tiles at the start of a
// stage), with the rounding the dx/dB walk's scaling applies to the same values.
__device__ __forceinline__ void bwd_scale_xdy(unsigned char* st, const float* gv, const float* fv,
                                              int ct) {
    uint4* xs = reinterpret_cast<uint4*>(st);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int idx = ct + kCT * i;  // 0..2047: [x h0 | x h1 | dy h0 | dy h1] 16-byte chunks
        const int k = ((idx >> 9) & 1) * 64 + ((idx >> 3) & 63);
        xs[idx] = scale_chunk(xs[idx], (idx < 1024) ? gv[k] : fv[k]);
    }
}

// Masked copy of a 64 x 64 M=64 accumulator (rows t in lanes 0..15 of each
// quadrant) into a K-major bf16 tile; keep (t, u) when (lower ? u <= t : u >= t).
// Every lane of the warp takes part: lane half hf holds columns 32 hf .. 32 hf + 31
// of row t.
__device__ __forceinline__ void masked_tile(uint32_t taddr_row, unsigned char* tile, int t,
                                            int hf, bool active, bool lower) {
    uint32_t v[32];
    tmem_ld16x2<32>(taddr_row + 0, &v[0]);
    tmem_ld16x2<32>(taddr_row + 16, &v[16]);
    tmem_wait_ld_regs<32>(v);
    if (!active) return;
    unsigned char* row = tile + t * 128;
#pragma unroll
    for (int e0 = 0; e0 < 32; e0 += 8) {
        const int e = 32 * hf + e0;
        float f[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const bool keep = lower ? (e + u <= t) : (e + u >= t);
            f[u] = keep ? __uint_as_float(v[e0 + u]) : 0.f;
        }
        *reinterpret_cast<uint4*>(row + ((((e >> 3) ^ t) & 7) << 4)) =
            make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]),
                       pack_bf16(f[6], f[7]));
    }
}

// masked_tile for the lower mask (u <= t) that also returns two sums over this thread's
// columns u <= t, with cb[u] = C_t . B_u in fp32 (zero past t):
//   .x = sum bf16(P[t, u]) cb[u]         (the tile as its MMA sees it, with exact C B^T),
//   .y = sum P[t, u] bf16(cb[u])         (fp32 P with the bf16 C B^T tile's values).
__device__ __forceinline__ float2 masked_tile_lower_dots(uint32_t taddr_row, unsigned char* tile,
                                                         int t, int hf, bool active,
                                                         const float* cb) {
    uint32_t v[32];
    tmem_ld16x2<32>(taddr_row + 0, &v[0]);
    tmem_ld16x2<32>(taddr_row + 16, &v[16]);
    tmem_wait_ld_regs<32>(v);
    if (!active) return make_float2(0.f, 0.f);
    unsigned char* row = tile + t * 128;
    float dr = 0.f, dc = 0.f;
#pragma unroll
    for (int e0 = 0; e0 < 32; e0 += 8) {
        const int e = 32 * hf + e0;
        float f[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) f[u] = (e + u <= t) ? __uint_as_float(v[e0 + u]) : 0.f;
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = pack_bf16(f[2 * i], f[2 * i + 1]);
        *reinterpret_cast<uint4*>(row + ((((e >> 3) ^ t) & 7) << 4)) =
            make_uint4(w[0], w[1], w[2], w[3]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 r = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
            const float2 l = __bfloat1622float2(__floats2bfloat162_rn(cb[e0 + 2 * i], cb[e0 + 2 * i + 1]));
            dr = fmaf(r.x, cb[e0 + 2 * i], dr);
            dr = fmaf(r.y, cb[e0 + 2 * i + 1], dr);
            dc = fmaf(f[2 * i], l.x, dc);
            dc = fmaf(f[2 * i + 1], l.y, dc);
        }
    }
    return make_float2(dr, dc);
}

// bf16(S) of this thread's row (h,p) and column half into the state operand buffer.
template <int NH>
__device__ __forceinline__ void write_state(unsigned char* sb, const float (&S)[NH], int r,
                                            int n0) {
    unsigned char* row = sb + r * 128;
#pragma unroll
    for (int c8 = 0; c8 < NH; c8 += 8) {
        const int n = n0 + c8;
        const uint4 v = make_uint4(pack_bf16(S[c8], S[c8 + 1]), pack_bf16(S[c8 + 2], S[c8 + 3]),
                                   pack_bf16(S[c8 + 4], S[c8 + 5]),
                                   pack_bf16(S[c8 + 6], S[c8 + 7]));
        *reinterpret_cast<uint4*>(row + (n >> 6) * 16384 + (((((n & 63) >> 3) ^ r) & 7) << 4)) = v;
    }
}

// Writes 16 fp32 values (columns n .. n+15 of row t) into the (N/32) x [64 x 32]
// fp32 staging tiles (128-byte swizzle, 16-byte chunk index XOR t % 8).
__device__ __forceinline__ void stage_row16(unsigned char* tiles, int t, int n, const float* v) {
    unsigned char* tile = tiles + (n >> 5) * 8192 + t * 128;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int chunk = ((n & 31) >> 2) + k;
        *reinterpret_cast<float4*>(tile + (((chunk ^ t) & 7) << 4)) =
            make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
    }
}

// ---------------------------------------------------------------- dC walk
template <int N>
__global__ void __launch_bounds__(kBwdThreads, 1)
    tc_bwd_dc_kernel(const __grid_constant__ CUtensorMap map_x,
                     const __grid_constant__ CUtensorMap map_dy,
                     const __grid_constant__ CUtensorMap map_b,
                     const __grid_constant__ CUtensorMap map_c,
                     const __grid_constant__ CUtensorMap map_acc, Args a) {
    using Lay = BwdLayout<N>;
    // pairs fastest: the CTAs that run together read whole token rows of x (and dy)
    const int seg = blockIdx.x / a.npairs;
    const int pr = blockIdx.x % a.npairs;
    const HeadPair hp = head_pair(a, pr);
    const int h0 = hp.h0;
    if (seg >= a.hdr->nseg) return;
    // an item beyond the factorisation's range: the dx/dB walk's SIMT evaluation adds dC
    if (a.fb[(long long)seg * a.npairs + pr]) return;
    const SegInfo si = a.segtab[seg];
    const int g = hp.g;
    const int nchunks = (si.len + kQ - 1) / kQ;
    // a sequence's last segment under an upstream final-state gradient: this walk also
    // forms the final state and writes <d final_state, final state> per head (kfin)
    const bool tail = (si.flags & SEG_LAST) && a.dhT != nullptr;

    extern __shared__ __align__(1024) unsigned char smraw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smraw) + 1023) & ~(uintptr_t)1023);
    ChunkFactors F;
    F.fbuf = reinterpret_cast<float*>(sm + Lay::OFF_F);
    F.gbuf = F.fbuf + 256;
    F.dbuf = F.gbuf + 256;
    F.scal = reinterpret_cast<float*>(sm + Lay::OFF_SC);
    F.red = reinterpret_cast<float*>(sm + Lay::OFF_RED);
    float* rpart = reinterpret_cast<float*>(sm + Lay::OFF_RQ);  // [2 wg][2 head][64]
    // [2 head][64]: ri_t - cs_t of the in-chunk sums below
    float* rint = reinterpret_cast<float*>(sm + Lay::OFF_RI);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Lay::OFF_BAR);
    uint64_t* full = bars + 0;      // [2]
    // [2] the chunk's partial dC tiles are in its stage, which the compute threads no
    // longer read (the producer adds them into the accumulator, then reloads the stage)
    uint64_t* staged = bars + 2;
    uint64_t* xg_ready = bars + 4;
    uint64_t* s_full = bars + 5;
    uint64_t* s_free = bars + 6;
    uint64_t* p1_full = bars + 7;
    uint64_t* w_ready = bars + 8;
    uint64_t* dc_full = bars + 10;
    uint64_t* dc_free = bars + 11;
    uint64_t* h_ready = bars + 12;  // [2], one per state operand buffer
    uint64_t* cb_full = bars + 14;  // the chunk's C B^T triangle landed
    uint64_t* cb_free = bars + 15;  // ... and was read by both compute warpgroups
    const float* cbt = reinterpret_cast<const float*>(sm + Lay::OFF_CB);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + Lay::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
    const uint32_t T_S = 0, T_P1 = 128, T_DC = 256;  // TMEM columns

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&staged[i], kCT);
        }
        mbar_init(xg_ready, kCT);
        mbar_init(s_full, 1);
        mbar_init(s_free, kCT);
        mbar_init(p1_full, 1);
        mbar_init(w_ready, kCT);
        mbar_init(&h_ready[0], kCT);
        mbar_init(&h_ready[1], kCT);
        mbar_init(dc_full, 1);
        mbar_init(dc_free, kCT);
        mbar_init(cb_full, 1);
        mbar_init(cb_free, kCT);
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
        if (lane == 0) {
            // partial dC tiles of chunk cc (in its stage) -> reduce-add into the accumulator
            auto add_partial = [&](int cc) -> bool {
                const int sc = cc & 1;
                if (!wait_or_abort(&staged[sc], (cc >> 1) & 1, abort_flag, a.hdr)) return false;
                unsigned char* rt = sm + Lay::OFF_STAGE + sc * Lay::STAGE;
                const int tok = (int)(si.start + (long long)cc * kQ);
                for (int j = 0; j < N / 32; ++j)
                    tma_reduce_add_3d(&map_acc, rt + j * 8192, j * 32, g, tok);
                tma_store_commit();
                return true;
            };
            bool run = true;
            for (int c = 0; c < nchunks && run; ++c) {
                const int s = c & 1;
                if (c >= 2) {
                    // the stage of chunk c - 2 is reloaded once its partial tiles are read
                    run = add_partial(c - 2);
                    tma_store_wait_read<0>();
                    if (!run) break;
                }
                unsigned char* st = sm + Lay::OFF_STAGE + s * Lay::STAGE;
                const int tok = (int)(si.start + (long long)c * kQ);
                mbar_expect_tx(&full[s], Lay::STAGE);
                tma_load_3d(st, &map_x, &full[s], 0, h0, tok);
                tma_load_3d(st + 8192, &map_x, &full[s], 0, hp.h1c, tok);
                tma_load_3d(st + 16384, &map_dy, &full[s], 0, h0, tok);
                tma_load_3d(st + 24576, &map_dy, &full[s], 0, hp.h1c, tok);
                for (int nb = 0; nb < N / 64; ++nb) {
                    tma_load_3d(st + 32768 + nb * 8192, &map_b, &full[s], nb * 64, g, tok);
                    tma_load_3d(st + 32768 + N * 128 + nb * 8192, &map_c, &full[s], nb * 64, g,
                                tok);
                }
                // the chunk's fp32 C B^T triangle, once the previous one has been read
                if (c >= 1 && !wait_or_abort(cb_free, (c - 1) & 1, abort_flag, a.hdr)) break;
                mbar_expect_tx(cb_full, kCbTri * 4);
                bulk_load(sm + Lay::OFF_CB,
                          a.cb32 + (((long long)seg * (a.Ls / kQ) + c) * a.G + g) * kCbTri,
                          kCbTri * 4, cb_full);
            }
            for (int cc = nchunks >= 2 ? nchunks - 2 : 0; cc < nchunks && run; ++cc)
                run = add_partial(cc);
            tma_store_wait_all<0>();
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t id_s = idesc_bf16(128, N, 1, 1);
            const uint32_t id_p = idesc_bf16(64, 64, 0, 0);
            const uint32_t id_c = idesc_bf16(64, N, 0, 1);
            for (int c = 0; c < nchunks; ++c) {
                const int s = c & 1, ph = (c >> 1) & 1, pc = c & 1;
                if (!wait_or_abort(&full[s], ph, abort_flag, a.hdr)) break;
                if (!wait_or_abort(xg_ready, pc, abort_flag, a.hdr)) break;
                if (c >= 1 && !wait_or_abort(s_free, pc ^ 1, abort_flag, a.hdr)) break;
                tc_fence_after();
                const uint32_t xs = smem_u32(sm + Lay::OFF_STAGE + s * Lay::STAGE);
                const uint32_t ys = xs + 16384, bs = xs + 32768;
                // chunk state, needed for later chunks and, with an upstream final-state
                // gradient, for the final state of a sequence's last segment
                if (c < nchunks - 1 || tail) {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_bf16(tmem + T_S, mdesc(xs, k, 8192), mdesc(bs, k, 8192), id_s,
                                 k > 0 ? 1u : 0u);
                }
                mma_commit(s_full);
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_bf16(tmem + T_P1 + h * 64, kdesc(ys + h * 8192, k, 0),
                                 kdesc(xs + h * 8192, k, 0), id_p, k > 0 ? 1u : 0u);
                mma_commit(p1_full);
                if (!wait_or_abort(w_ready, pc, abort_flag, a.hdr)) break;
                if (!wait_or_abort(&h_ready[s], ph, abort_flag, a.hdr)) break;
                if (c >= 1 && !wait_or_abort(dc_free, pc ^ 1, abort_flag, a.hdr)) break;
                tc_fence_after();
                const uint32_t wt = smem_u32(sm + Lay::OFF_T0);
                const uint32_t hb = smem_u32(sm + Lay::OFF_S + s * Lay::SBUF);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_bf16(tmem + T_DC + h * N, kdesc(wt + h * 8192, k, 0),
                                 mdesc(bs, k, 8192), id_c, k > 0 ? 1u : 0u);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_bf16(tmem + T_DC + h * N, kdesc(ys + h * 8192, k, 0),
                                 mdesc(hb + h * 8192, k, 16384), id_c, 1u);
                }
                mma_commit(dc_full);
            }
        }
    } else {
        const int ct = tid - 64;
        const int wg = ct >> 7;
        const int q = warp & 3;
        const int r = 32 * q + lane;        // M=128 row (h, p)
        const int rh = r >> 6, rp = r & 63;
        const int t = 16 * q + (lane & 15);  // M=64 row (token)
        const int hf = lane >> 4;            // M=64 column half of this lane
        constexpr int NH = N / 2;
        const int n0 = wg * NH;
        const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16);
        float Hs[NH];

        bwd_factors(F, load_fac_vals(a, seg, pr, 0, nchunks, ct), 0, ct);
        {
            // a dummy second slot starts (and stays) at zero
            const float sc0 = (rh == 0 || hp.v1) ? expf(-F.scal[(0 * 2 + rh) * 4 + 0]) : 0.f;
            const float* Hin = a.A + ((long long)seg * a.H + h0 + (hp.v1 ? rh : 0)) * kP * N +
                               lm_row(rp, N) + n0 * 32;
#pragma unroll
            for (int i = 0; i < NH; i += 4) {
                const float4 v = *reinterpret_cast<const float4*>(Hin + i * 32);
                Hs[i] = v.x * sc0;
                Hs[i + 1] = v.y * sc0;
                Hs[i + 2] = v.z * sc0;
                Hs[i + 3] = v.w * sc0;
            }
        }
        write_state<NH>(sm + Lay::OFF_S, Hs, r, n0);
        fence_proxy_async();
        mbar_arrive(&h_ready[0]);
        // x -> g x and dy -> f dy of chunk cc in its stage (factors in buffer cc & 1): the
        // dx/dB walk forms q from the same bf16 f dy, which the in-chunk sums below need
        auto scale_chunk_stage = [&](int cc) {
            const int sc = cc & 1;
            if (wait_or_abort(&full[sc], (cc >> 1) & 1, abort_flag, a.hdr))
                bwd_scale_xdy(sm + Lay::OFF_STAGE + sc * Lay::STAGE, F.gbuf + sc * 128,
                              F.fbuf + sc * 128, ct);
            fence_proxy_async();
            mbar_arrive(xg_ready);
        };
        scale_chunk_stage(0);

        for (int c = 0; c < nchunks; ++c) {
            const int s = c & 1, pc = c & 1;
            const bool last = (c == nchunks - 1);
            const int vc = min(kQ, si.len - c * kQ);
            const long long tok0 = si.start + (long long)c * kQ;
            unsigned char* st = sm + Lay::OFF_STAGE + s * Lay::STAGE;
            const FacVals fac_next = load_fac_vals(a, seg, pr, c + 1, nchunks, ct);
            // B: W_h = P1_h masked to s <= t (warpgroup h handles head h), and two in-chunk
            // sums of row t for the delta gradient:
            //   ri_t = sum_s W_h[t, s] C_t . B_s, the part of r_t from the chunk's own tokens
            //          as the dC MMA gives it (bf16 W_h, exact products), and
            //   cs_t = sum_s P1_h[t, s] L0[t, s], the same pairs as the dx/dB walk's DX MMA
            //          gives them (fp32 products of the bf16 f dy, g x and L0 values).
            // r_t - ri_t + cs_t is stored: summed over u >= t it leaves, up to fp32 rounding,
            // the in-chunk pairs s < t <= u that the delta gradient needs, instead of the
            // difference of two differently rounded sums of every in-chunk pair.
            {
                bool ok = wait_or_abort(cb_full, pc, abort_flag, a.hdr);
                // row t of the triangle, columns 32 hf .. 32 hf + 31 (those past t are
                // masked; the index stays inside the triangle for every t)
                float cbv[32];
                const float* crow = cbt + cb_tri_row(t) + 32 * hf;
#pragma unroll
                for (int j = 0; j < 32; ++j) cbv[j] = (32 * hf + j <= t) ? crow[j] : 0.f;
                mbar_arrive(cb_free);
                ok = wait_or_abort(p1_full, pc, abort_flag, a.hdr) && ok;
                tc_fence_after();
                const float2 dots = masked_tile_lower_dots(tq + T_P1 + wg * 64,
                                                           sm + Lay::OFF_T0 + wg * 8192, t, hf,
                                                           ok, cbv);
                fence_proxy_async();
                mbar_arrive(w_ready);
                const float dd = dots.x - dots.y;
                const float dsum = dd + __shfl_xor_sync(0xffffffffu, dd, 16);  // whole warp
                if (hf == 0) rint[wg * 64 + t] = dsum;
            }
            // C: chunk state -> Hs for the next chunk (kept in registers until dC is done)
            if (!last) {
                bwd_factors(F, fac_next, c + 1, ct);
                const bool ok = wait_or_abort(s_full, pc, abort_flag, a.hdr);
                tc_fence_after();
                const float gam = expf(-(F.scal[(s * 2 + rh) * 4] + F.scal[((s ^ 1) * 2 + rh) * 4]));
#pragma unroll
                for (int c0 = 0; c0 < NH; c0 += 32) {
                    uint32_t v[32];
                    tmem_ld16(tq + T_S + n0 + c0, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
                    tmem_ld16(tq + T_S + n0 + c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
                    tmem_wait_ld_regs<32>(v);
                    if (ok) {
#pragma unroll
                        for (int u = 0; u < 32; ++u) Hs[c0 + u] = gam * (Hs[c0 + u] + __uint_as_float(v[u]));
                    }
                }
                tc_fence_before();
                mbar_arrive(s_free);
                // the next chunk's state operand, in the other buffer (dC of chunk c - 1,
                // its previous reader, completed before this iteration's epilogue)
                write_state<NH>(sm + Lay::OFF_S + (s ^ 1) * Lay::SBUF, Hs, r, n0);
                fence_proxy_async();
                mbar_arrive(&h_ready[s ^ 1]);
            } else if (tail) {
                // final state = exp(-half_c) (Hs_c + S_c) (the chain's update with no next
                // chunk), dotted with the upstream gradient of the final state
                const bool ok = wait_or_abort(s_full, pc, abort_flag, a.hdr);
                tc_fence_after();
                const float gend = expf(-F.scal[(s * 2 + rh) * 4]);
                const float* dT =
                    a.dhT + (((long long)si.seq * a.H + h0 + (hp.v1 ? rh : 0)) * kP + rp) * N + n0;
                float kp = 0.f;
#pragma unroll
                for (int c0 = 0; c0 < NH; c0 += 32) {
                    uint32_t v[32];
                    tmem_ld16(tq + T_S + n0 + c0, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
                    tmem_ld16(tq + T_S + n0 + c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
                    tmem_wait_ld_regs<32>(v);
#pragma unroll
                    for (int u = 0; u < 32; u += 4) {
                        const float4 d4 = *reinterpret_cast<const float4*>(dT + c0 + u);
                        kp = fmaf(gend * (Hs[c0 + u] + __uint_as_float(v[u])), d4.x, kp);
                        kp = fmaf(gend * (Hs[c0 + u + 1] + __uint_as_float(v[u + 1])), d4.y, kp);
                        kp = fmaf(gend * (Hs[c0 + u + 2] + __uint_as_float(v[u + 2])), d4.z, kp);
                        kp = fmaf(gend * (Hs[c0 + u + 3] + __uint_as_float(v[u + 3])), d4.w, kp);
                    }
                }
                tc_fence_before();
                mbar_arrive(s_free);
                kp = warp_sum(kp);
                if (lane == 0) F.red[wg * 4 + q] = (ok && (rh == 0 || hp.v1)) ? kp : 0.f;
                named_sync(1, kCT);
                // quadrants 0-1 hold head 0, 2-3 head 1; both warpgroups hold column halves
                if (ct < (hp.v1 ? 2 : 1))
                    a.kfin[(long long)seg * a.H + h0 + ct] =
                        (F.red[2 * ct] + F.red[2 * ct + 1]) + (F.red[4 + 2 * ct] + F.red[5 + 2 * ct]);
            } else {
                mbar_arrive(s_free);
            }
            // A for the next chunk: scaled now, so that its S and P1 MMAs run during this
            // chunk's epilogue
            if (!last) scale_chunk_stage(c + 1);
            // D: dC rows (both heads, this warpgroup's column half split over the two lane
            // halves), r partials
            {
                const bool ok = wait_or_abort(dc_full, pc, abort_flag, a.hdr);
                tc_fence_after();
                const unsigned char* cst = st + 32768 + N * 128;
                float rp0 = 0.f, rp1 = 0.f;
                // the partial dC tiles go into this stage's x / dy tiles, which every MMA of
                // the chunk has finished reading
                unsigned char* rtiles = st;
#pragma unroll
                for (int c0 = 0; c0 < NH / 2; c0 += 16) {
                    const int n = n0 + (NH / 2) * hf + c0;
                    uint32_t v0[16], v1[16];
                    tmem_ld16x2<NH / 2>(tq + T_DC + n0 + c0, v0);
                    tmem_ld16x2<NH / 2>(tq + T_DC + N + n0 + c0, v1);
                    tmem_wait_ld_regs<16>(v0);
                    reg_dep16(v1);
                    if (ok) {
                        const unsigned char* crow = cst + (n >> 6) * 8192 + t * 128;
                        float cv[16];
#pragma unroll
                        for (int e = 0; e < 16; e += 8) {
                            const uint4 w = *reinterpret_cast<const uint4*>(
                                crow + (((((n & 63) + e) >> 3) ^ t) & 7) * 16);
                            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const float2 f2 = __bfloat1622float2(
                                    *reinterpret_cast<const __nv_bfloat162*>(&ww[i]));
                                cv[e + 2 * i] = f2.x;
                                cv[e + 2 * i + 1] = f2.y;
                            }
                        }
#pragma unroll
                        for (int u = 0; u < 16; ++u) {
                            const float d0 = __uint_as_float(v0[u]), d1 = __uint_as_float(v1[u]);
                            rp0 = fmaf(cv[u], d0, rp0);
                            rp1 = fmaf(cv[u], d1, rp1);
                        }
                    }
                    {  // partial dC (both heads); rows past the chunk's tokens add zero
                        float sum[16];
#pragma unroll
                        for (int u = 0; u < 16; ++u)
                            sum[u] = (ok && t < vc) ? __uint_as_float(v0[u]) + __uint_as_float(v1[u])
                                                    : 0.f;
                        stage_row16(rtiles, t, n, sum);
                    }
                }
                rp0 += __shfl_xor_sync(0xffffffffu, rp0, 16);
                rp1 += __shfl_xor_sync(0xffffffffu, rp1, 16);
                tc_fence_before();
                mbar_arrive(dc_free);
                fence_proxy_async();
                mbar_arrive(&staged[s]);
                if (hf == 0) {
                    rpart[(wg * 2 + 0) * 64 + t] = rp0;
                    rpart[(wg * 2 + 1) * 64 + t] = rp1;
                }
                named_sync(1, kCT);
                if (wg == 0 && hf == 0 && t < vc && ok) {
                    a.rtok[(tok0 + t) * a.H + h0] =
                        (rpart[0 * 64 + t] + rpart[2 * 64 + t]) - rint[t];
                    if (hp.v1)
                        a.rtok[(tok0 + t) * a.H + h0 + 1] =
                            (rpart[1 * 64 + t] + rpart[3 * 64 + t]) - rint[64 + t];
                }
            }
            named_sync(1, kCT);  // rpart reuse
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------- dX / dB walk
// Chunks in reverse order.  Warps: 0 = TMA producer (x, dy, B, C; the chunk's L0 tile
// and factor records), 1 = MMA issuer of S' and P2, 18 = MMA issuer of DX and dB,
// 2..17 = four compute warpgroups with one task each:
//   warpgroup 0     x -> g x and dy -> f dy in place, one chunk ahead;
//   warpgroup 1     the masked P2 tiles, then dx = g DX, q = xg . DX and d_raw;
//   warpgroups 2-3  the adjoint chain in TMEM (S' accumulates onto Gs there; these
//                   warps rescale it by gamma), its bf16 operand, and the partial dB
//                   tiles, added into the fp32 accumulator by TMA reduce-add.
constexpr int kDxThreads = 64 + 4 * 128 + 32;
constexpr int kDFS = 4;  // factor record slots (processing index it uses slot it % kDFS)

template <int N>
struct DxLayout {
    static constexpr int STAGE = 32768 + 2 * N * 128;       // x h0 | x h1 | dy h0 | dy h1 | B | C
    static constexpr int OFF_STAGE = 0;
    static constexpr int OFF_P2M = 2 * STAGE;                // masked P2, 2 x 8K
    static constexpr int OFF_L0 = OFF_P2M + 16384;           // L0 tile (read as L0^T), 8K
    static constexpr int OFF_G = OFF_L0 + 8192;              // bf16 Gs operand, (N/64) x 16K
    static constexpr int OFF_DB = OFF_G + (N / 64) * 16384;  // fp32 dB staging, (N/32) x 8K
    static constexpr int OFF_F = OFF_DB + N * 256;           // factor records [slot][head]
    static constexpr int OFF_RQ = OFF_F + kDFS * kFSlot;          // [2 head][4 quadrant]
    static constexpr int OFF_RED = OFF_RQ + 64;                   // [16]
    static constexpr int OFF_BAR = OFF_RED + 64;
    static constexpr int NBAR = 40;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int TOTAL = OFF_MISC + 16 + 1024;
};

template <int N>
__global__ void __launch_bounds__(kDxThreads, 1)
    tc_bwd_dxdb_kernel(const __grid_constant__ CUtensorMap map_x,
                       const __grid_constant__ CUtensorMap map_dy,
                       const __grid_constant__ CUtensorMap map_b,
                       const __grid_constant__ CUtensorMap map_c,
                       const __grid_constant__ CUtensorMap map_acc, Args a) {
    using Lay = DxLayout<N>;
    // pairs fastest: the CTAs that run together read whole token rows of x (and dy)
    const int seg = blockIdx.x / a.npairs;
    const int pr = blockIdx.x % a.npairs;
    const HeadPair hpr = head_pair(a, pr);
    const int h0 = hpr.h0;
    if (seg >= a.hdr->nseg) return;
    if (a.fb[(long long)seg * a.npairs + pr]) {
        // a chunk decay beyond the factorisation's range: the SIMT recurrence for both heads
        // (dx, dB and dC added into the accumulators, the finished d_raw_dt)
        extern __shared__ float fsm[];
        if (threadIdx.x < simt::kSimtThreads) fallback_bwd<N>(a, seg, pr, fsm, 10);
        return;
    }
    const SegInfo si = a.segtab[seg];
    const int g = hpr.g;
    const int nchunks = (si.len + kQ - 1) / kQ;

    extern __shared__ __align__(1024) unsigned char smraw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smraw) + 1023) & ~(uintptr_t)1023);
    // factor record of (slot, head): f[64], g[64], delta[64], half
    auto frec = [&](int sl, int head) -> const float* {
        return reinterpret_cast<const float*>(sm + Lay::OFF_F + sl * kFSlot) + head * kFacRec;
    };
    float* rqs = reinterpret_cast<float*>(sm + Lay::OFF_RQ);   // [2 head][4]
    float* red = reinterpret_cast<float*>(sm + Lay::OFF_RED);  // 8..15: kseg partials
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Lay::OFF_BAR);
    uint64_t* full = bars + 0;        // [2] stage landed
    uint64_t* empty = bars + 2;       // [2] stage read by the MMAs and by the q epilogue
    uint64_t* xg_ready = bars + 4;    // [2] x, dy scaled in place (warpgroup 0)
    uint64_t* l0_full = bars + 6;     // L0 tile landed
    uint64_t* l0_free = bars + 7;     // DX has read the L0 tile
    uint64_t* s_full = bars + 8;      // S' accumulated onto Gs
    uint64_t* s_free = bars + 9;      // Gs rescaled in TMEM (state warps)
    uint64_t* p2_full = bars + 10;    // P2 accumulated
    uint64_t* e_ready = bars + 11;    // P2 read from TMEM and masked into P2M (warpgroup 1)
    uint64_t* p2m_free = bars + 12;   // dB has read P2M
    uint64_t* g_ready = bars + 13;    // bf16 Gs operand written (state warps)
    uint64_t* g_free = bars + 14;     // DX and dB have read the Gs operand
    uint64_t* dx_full = bars + 15;    // DX accumulated
    uint64_t* dx_free = bars + 16;    // DX read (warpgroup 1)
    uint64_t* db_full = bars + 17;    // dB accumulated
    uint64_t* db_free = bars + 18;    // dB read (state warps)
    uint64_t* kseg_ready = bars + 19; // boundary term written (state warps)
    uint64_t* fac_full = bars + 20;   // [kDFS]
    uint64_t* fac_empty = bars + 24;  // [kDFS]
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + Lay::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
    // TMEM columns: Gs (+ S') 0..127, P2 128..255 (2 x 64), DX 256..383, dB 384..511
    const uint32_t T_G = 0, T_P2 = 128, T_DX = 256, T_DB = 384;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1 + 128);
            mbar_init(&xg_ready[i], 128);
        }
        mbar_init(l0_full, 1);
        mbar_init(l0_free, 1);
        mbar_init(s_full, 1);
        mbar_init(s_free, 256);
        mbar_init(p2_full, 1);
        mbar_init(e_ready, 128);
        mbar_init(p2m_free, 1);
        mbar_init(g_ready, 256);
        mbar_init(g_free, 1);
        mbar_init(dx_full, 1);
        mbar_init(dx_free, 128);
        mbar_init(db_full, 1);
        mbar_init(db_free, 256);
        mbar_init(kseg_ready, 256);
        for (int i = 0; i < kDFS; ++i) {
            mbar_init(&fac_full[i], 1);
            mbar_init(&fac_empty[i], 128 + 128 + 256);
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
            const int cps = a.Ls / kQ;
            // the factor records of processing index j (both heads) into slot j % kDFS
            auto load_fac = [&](int j) {
                const int fs = j % kDFS, cc = nchunks - 1 - j;
                mbar_expect_tx(&fac_full[fs], kFSlot);
                bulk_load(sm + Lay::OFF_F + fs * kFSlot,
                          a.fac + ((long long)(seg * cps + cc) * a.Hf + 2 * pr) * kFacRec, kFSlot,
                          &fac_full[fs]);
            };
            for (int j = 0; j < 2 && j < nchunks; ++j) load_fac(j);
            for (int it = 0; it < nchunks; ++it) {
                const int c = nchunks - 1 - it, s = it & 1;
                if (it >= 2 && !wait_or_abort(&empty[s], ((it >> 1) - 1) & 1, abort_flag, a.hdr))
                    break;
                unsigned char* st = sm + Lay::OFF_STAGE + s * Lay::STAGE;
                const int tok = (int)(si.start + (long long)c * kQ);
                mbar_expect_tx(&full[s], Lay::STAGE);
                tma_load_3d(st, &map_x, &full[s], 0, h0, tok);
                tma_load_3d(st + 8192, &map_x, &full[s], 0, hpr.h1c, tok);
                tma_load_3d(st + 16384, &map_dy, &full[s], 0, h0, tok);
                tma_load_3d(st + 24576, &map_dy, &full[s], 0, hpr.h1c, tok);
                for (int nb = 0; nb < N / 64; ++nb) {
                    tma_load_3d(st + 32768 + nb * 8192, &map_b, &full[s], nb * 64, g, tok);
                    tma_load_3d(st + 32768 + N * 128 + nb * 8192, &map_c, &full[s], nb * 64, g,
                                tok);
                }
                if (it >= 1 && !wait_or_abort(l0_free, (it - 1) & 1, abort_flag, a.hdr)) break;
                mbar_expect_tx(l0_full, 8192);
                bulk_load(sm + Lay::OFF_L0, a.l0 + (((long long)seg * cps + c) * a.G + g) * 8192,
                          8192, l0_full);
                const int jf = it + 2;
                if (jf < nchunks) {
                    if (jf >= kDFS && !wait_or_abort(&fac_empty[jf % kDFS], ((jf / kDFS) - 1) & 1,
                                                     abort_flag, a.hdr))
                        break;
                    load_fac(jf);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer: S', P2
        if (lane == 0) {
            const uint32_t id_p2 = idesc_bf16(64, 64, 0, 0);
            const uint32_t id_sp = idesc_bf16(128, N, 1, 1);
            for (int it = 0; it < nchunks; ++it) {
                const int s = it & 1, ph = (it >> 1) & 1;
                if (!wait_or_abort(&xg_ready[s], ph, abort_flag, a.hdr)) break;
                const uint32_t xs = smem_u32(sm + Lay::OFF_STAGE + s * Lay::STAGE);
                const uint32_t ys = xs + 16384, cs = xs + 32768 + N * 128;
                // S' = dyf^T C onto Gs (not needed for the segment's first chunk)
                if (it < nchunks - 1) {
                    if (!wait_or_abort(s_free, it & 1, abort_flag, a.hdr)) break;
                    tc_fence_after();
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_bf16(tmem + T_G, mdesc(ys, k, 8192), mdesc(cs, k, 8192), id_sp, 1u);
                    mma_commit(s_full);
                }
                // P2_h = xg_h dyf_h^T, once warpgroup 1 has read the previous P2
                if (it >= 1 && !wait_or_abort(e_ready, (it - 1) & 1, abort_flag, a.hdr)) break;
                tc_fence_after();
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_bf16(tmem + T_P2 + h * 64, kdesc(xs + h * 8192, k, 0),
                                 kdesc(ys + h * 8192, k, 0), id_p2, k > 0 ? 1u : 0u);
                mma_commit(p2_full);
            }
        }
    } else if (warp == 18) {
        // ------------------------------------------------ MMA issuer: DX, dB
        if (lane == 0) {
            const uint32_t id_dx1 = idesc_bf16(64, 128, 1, 1);
            const uint32_t id_dx2 = idesc_bf16(64, 128, 0, 0);
            const uint32_t id_db = idesc_bf16(64, N, 0, 1);
            const uint32_t l0 = smem_u32(sm + Lay::OFF_L0);
            const uint32_t p2m = smem_u32(sm + Lay::OFF_P2M);
            const uint32_t gb = smem_u32(sm + Lay::OFF_G);
            for (int it = 0; it < nchunks; ++it) {
                const int s = it & 1, ph = (it >> 1) & 1;
                if (!wait_or_abort(&xg_ready[s], ph, abort_flag, a.hdr)) break;
                if (!wait_or_abort(g_ready, it & 1, abort_flag, a.hdr)) break;
                if (!wait_or_abort(l0_full, it & 1, abort_flag, a.hdr)) break;
                if (it >= 1 && !wait_or_abort(dx_free, (it - 1) & 1, abort_flag, a.hdr)) break;
                tc_fence_after();
                const uint32_t xs = smem_u32(sm + Lay::OFF_STAGE + s * Lay::STAGE);
                const uint32_t ys = xs + 16384, bs = xs + 32768, cs = bs + N * 128;
                // DX = L0^T dyf + B Gs^T
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_bf16(tmem + T_DX, mdesc(l0, k, 0), mdesc(ys, k, 8192), id_dx1,
                             k > 0 ? 1u : 0u);
#pragma unroll
                for (int k = 0; k < N / 16; ++k)
                    mma_bf16(tmem + T_DX, kdesc(bs, k, 8192), kdesc(gb, k, 16384), id_dx2, 1u);
                mma_commit(dx_full);
                mma_commit(l0_free);
                // dB = sum_h xg_h Gs_h + P2m_h C: the first half needs no masks and is the
                // last reader of the Gs operand
                if (it >= 1 && !wait_or_abort(db_free, (it - 1) & 1, abort_flag, a.hdr)) break;
                tc_fence_after();
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_bf16(tmem + T_DB, kdesc(xs + h * 8192, k, 0),
                                 mdesc(gb + h * 8192, k, 16384), id_db, (h > 0 || k > 0) ? 1u : 0u);
                mma_commit(g_free);
                if (!wait_or_abort(e_ready, it & 1, abort_flag, a.hdr)) break;
                tc_fence_after();
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_bf16(tmem + T_DB, kdesc(p2m + h * 8192, k, 0), mdesc(cs, k, 8192),
                                 id_db, 1u);
                mma_commit(db_full);
                mma_commit(p2m_free);
                mma_commit(&empty[s]);
            }
        }
    } else {
        const int ct = tid - 64;  // 0..511
        const int wg = ct >> 7;
        const int q = warp & 3;
        const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16);
        const int tt = 16 * q + (lane & 15);  // M=64 accumulator row (token)
        const int hf = lane >> 4;             // M=64 column half of this lane
        if (wg == 0) {
            // ------------------------------------------------ scaling
            // x -> g x, dy -> f dy for processing index j (one chunk ahead of the masks)
            auto scale = [&](int j) {
                const int s = j & 1, fs = j % kDFS;
                bool ok = wait_or_abort(&fac_full[fs], (j / kDFS) & 1, abort_flag, a.hdr);
                ok = wait_or_abort(&full[s], (j >> 1) & 1, abort_flag, a.hdr) && ok;
                if (ok) {
                    uint4* xs = reinterpret_cast<uint4*>(sm + Lay::OFF_STAGE + s * Lay::STAGE);
                    // two chunks in flight per thread: a deeper unroll makes this warpgroup
                    // crowd the shared-memory pipe that the masks and epilogues wait on (measured
                    // slower at 4 and 16)
#pragma unroll 2
                    for (int i = 0; i < 16; ++i) {
                        const int idx = ct + 128 * i;  // [x h0 | x h1 | dy h0 | dy h1] 16-byte chunks
                        const int tile = idx >> 9, row = (idx >> 3) & 63;
                        const float* rec = frec(fs, tile & 1);
                        xs[idx] = scale_chunk(xs[idx], (tile < 2) ? rec[FAC_G + row] : rec[FAC_F + row]);
                    }
                }
                fence_proxy_async();
                mbar_arrive(&xg_ready[s]);
                mbar_arrive(&fac_empty[fs]);
            };
            for (int j = 0; j < nchunks; ++j) scale(j);
        } else if (wg == 1) {
            // ------------------------------------------------ P2 masks, dx, d_raw
            // thread (token tt, head hf)
            const float* rtok = a.rtok;
            float carry = 0.f;  // sum of (r - q) over the later chunks of the segment, head hf
            wait_or_abort(kseg_ready, 0, abort_flag, a.hdr);
            // a sequence's last segment: <d final_state, final state>, from the dC walk
            const float kseg = ((si.flags & SEG_LAST) && a.dhT)
                                   ? ((hf == 0 || hpr.v1) ? a.kfin[(long long)seg * a.H + h0 + hf] : 0.f)
                                   : (red[8 + 2 * hf] + red[9 + 2 * hf]) +
                                         (red[12 + 2 * hf] + red[13 + 2 * hf]);
            for (int it = 0; it < nchunks; ++it) {
                const int c = nchunks - 1 - it;
                const int s = it & 1, sl = it % kDFS;
                const int vc = min(kQ, si.len - c * kQ);
                const long long tok0 = si.start + (long long)c * kQ;
                const bool real = hf == 0 || hpr.v1;  // this thread's head slot holds a head
                const float rv = (tt < vc && real) ? rtok[(tok0 + tt) * a.H + h0 + hf] : 0.f;
                {
                // P2 of both heads masked to u >= t, bf16 into P2M once dB of the previous
                // chunk has read it (thread (token tt, column half hf) of each tile)
                bool okm = wait_or_abort(p2_full, it & 1, abort_flag, a.hdr);
                if (it >= 1) okm = wait_or_abort(p2m_free, (it - 1) & 1, abort_flag, a.hdr) && okm;
                tc_fence_after();
                masked_tile(tq + T_P2, sm + Lay::OFF_P2M, tt, hf, okm, false);
                masked_tile(tq + T_P2 + 64, sm + Lay::OFF_P2M + 8192, tt, hf, okm, false);
                tc_fence_before();
                fence_proxy_async();
                mbar_arrive(e_ready);
                }
                // dx = g DX and q = xg . DX for (token tt, head hf)
                bool ok = wait_or_abort(&fac_full[sl], (it / kDFS) & 1, abort_flag, a.hdr);
                ok = wait_or_abort(dx_full, it & 1, abort_flag, a.hdr) && ok;
                tc_fence_after();
                const float gt = frec(sl, hf)[FAC_G + tt];
                const float dt = frec(sl, hf)[FAC_D + tt];
                mbar_arrive(&fac_empty[sl]);
                const unsigned char* xrow =
                    sm + Lay::OFF_STAGE + s * Lay::STAGE + hf * 8192 + tt * 128;  // xg, row tt
                __nv_bfloat16* dxrow =
                    static_cast<__nv_bfloat16*>(a.dx) + ((tok0 + tt) * a.H + h0 + hf) * kP;
                float qv = 0.f;
#pragma unroll
                for (int j = 0; j < 64; j += 32) {
                    uint32_t v[32];
                    tmem_ld16x2<64>(tq + T_DX + j, &v[0]);
                    tmem_ld16x2<64>(tq + T_DX + j + 16, &v[16]);
                    tmem_wait_ld_regs<32>(v);
                    if (j == 32) {
                        tc_fence_before();
                        mbar_arrive(dx_free);
                    }
                    if (ok) {
#pragma unroll
                        for (int e = 0; e < 32; e += 8) {
                            const uint4 w = *reinterpret_cast<const uint4*>(
                                xrow + ((((j + e) >> 3) ^ tt) & 7) * 16);
                            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const float2 xf = __bfloat1622float2(
                                    *reinterpret_cast<const __nv_bfloat162*>(&ww[i]));
                                qv = fmaf(xf.x, __uint_as_float(v[e + 2 * i]), qv);
                                qv = fmaf(xf.y, __uint_as_float(v[e + 2 * i + 1]), qv);
                            }
                        }
                    }
                    // this warpgroup is done with the stage's xg rows
                    if (j == 32) mbar_arrive(&empty[s]);
                    if (ok) {
                        if (tt < vc && real) {
#pragma unroll
                            for (int e = 0; e < 32; e += 8)
                                *reinterpret_cast<uint4*>(dxrow + j + e) = make_uint4(
                                    pack_bf16(gt * __uint_as_float(v[e]), gt * __uint_as_float(v[e + 1])),
                                    pack_bf16(gt * __uint_as_float(v[e + 2]), gt * __uint_as_float(v[e + 3])),
                                    pack_bf16(gt * __uint_as_float(v[e + 4]), gt * __uint_as_float(v[e + 5])),
                                    pack_bf16(gt * __uint_as_float(v[e + 6]), gt * __uint_as_float(v[e + 7])));
                        }
                    }
                }
                // d_raw = sigmoid(z) (q / delta - sum_{u >= t in the segment} (r - q) - kseg):
                // suffix sums over the chunk's rows u >= t (16 rows per warp and head, then
                // the later warps' totals), plus the later chunks' carry
                const float xgb = (dt > 1e-30f) ? qv / dt : 0.f;
                float suf = (ok && tt < vc) ? (rv - qv) : 0.f;
#pragma unroll
                for (int o = 1; o < 16; o <<= 1) {
                    const float nb = __shfl_down_sync(0xffffffffu, suf, o, 16);
                    if ((lane & 15) + o < 16) suf += nb;
                }
                if ((lane & 15) == 0) rqs[hf * 4 + q] = suf;
                named_sync(6, 128);
                float later = 0.f, tot = 0.f;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float x = rqs[hf * 4 + k];
                    tot += x;
                    if (k > q) later += x;
                }
                named_sync(6, 128);  // rqs is rewritten by the next chunk
                suf += later;
                if (ok && tt < vc && real)
                    a.draw[(tok0 + tt) * a.H + h0 + hf] =
                        -expm1f(-dt) * (xgb - (carry + suf + kseg));
                carry += tot;
            }
        } else {
            // ------------------------------------------------ adjoint chain, dB tiles
            // Gs rows r = (head, p), columns [n0, n0 + N / 2) of this warpgroup; the state is
            // kept as Gs_c = exp(s_end - m_c) G_c and rewritten in TMEM as
            //   Gs_{c-1} = exp(-(half_c + half_{c-1})) (Gs_c + S'_c)
            constexpr int NH = N / 2;
            const int sct = ct - 256;         // 0..255
            const int r = 32 * q + lane;
            const int rh = r >> 6, rp = r & 63;
            const int n0 = (wg - 2) * NH;
            const uint32_t tcol = tq + T_G + n0;
            uint32_t hp[NH / 2];  // bf16 pairs of the next chunk's operand
            auto write_g = [&]() {
                unsigned char* row = sm + Lay::OFF_G + r * 128;
#pragma unroll
                for (int c8 = 0; c8 < NH; c8 += 8) {
                    const int n = n0 + c8;
                    *reinterpret_cast<uint4*>(row + (n >> 6) * 16384 +
                                              (((((n & 63) >> 3) ^ r) & 7) << 4)) =
                        make_uint4(hp[c8 / 2], hp[c8 / 2 + 1], hp[c8 / 2 + 2], hp[c8 / 2 + 3]);
                }
                fence_proxy_async();
                mbar_arrive(g_ready);
            };
            {
                // adjoint arriving at the segment end, and kseg = <G_seg, H_end>: the pairs of
                // the quadratic form with one end in or before this segment and the other
                // after it (both states from the fp32 scans)
                wait_or_abort(&fac_full[0], 0, abort_flag, a.hdr);
                // a dummy second slot starts (and stays) at zero, with no boundary term
                const bool realr = rh == 0 || hpr.v1;
                const float sc = realr ? expf(-frec(0, rh)[FAC_HALF]) : 0.f;
                const float* Gin = a.adj + ((long long)seg * a.H + h0 + (hpr.v1 ? rh : 0)) * kP * N +
                                   lm_row(rp, N) + n0 * 32;
                const bool more = !(si.flags & SEG_LAST) && realr;
                const float* Hend = a.A + ((long long)(seg + 1) * a.H + h0 + (hpr.v1 ? rh : 0)) * kP * N +
                                    lm_row(rp, N) + n0 * 32;
                float kp = 0.f;
#pragma unroll
                for (int c0 = 0; c0 < NH; c0 += 16) {
                    float h[16];
#pragma unroll
                    for (int i = 0; i < 16; i += 4) {
                        const float4 v = *reinterpret_cast<const float4*>(Gin + (c0 + i) * 32);
                        if (more) {
                            const float4 w = *reinterpret_cast<const float4*>(Hend + (c0 + i) * 32);
                            kp += v.x * w.x + v.y * w.y + v.z * w.z + v.w * w.w;
                        }
                        h[i] = v.x * sc;
                        h[i + 1] = v.y * sc;
                        h[i + 2] = v.z * sc;
                        h[i + 3] = v.w * sc;
                    }
                    tmem_st16(tcol + c0, reinterpret_cast<const uint32_t*>(h));
#pragma unroll
                    for (int i = 0; i < 16; i += 2) hp[(c0 + i) / 2] = pack_bf16(h[i], h[i + 1]);
                }
                kp = warp_sum(kp);
                if (lane == 0) red[8 + (wg - 2) * 4 + q] = kp;  // partial of head q / 2
                mbar_arrive(kseg_ready);
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(s_free);
                write_g();
            }
            for (int it = 0; it < nchunks; ++it) {
                const int c = nchunks - 1 - it;
                const int sl = it % kDFS, sn = (it + 1) % kDFS;
                const long long tok0 = si.start + (long long)c * kQ;
                const int vc = min(kQ, si.len - c * kQ);
                const bool more = it + 1 < nchunks;
                // (a) Gs of the next chunk, in TMEM and as bf16 pairs in registers
                if (more) {
                    bool ok = wait_or_abort(&fac_full[sn], ((it + 1) / kDFS) & 1, abort_flag, a.hdr);
                    const float gam = expf(-(frec(sl, rh)[FAC_HALF] + frec(sn, rh)[FAC_HALF]));
                    ok = wait_or_abort(s_full, it & 1, abort_flag, a.hdr) && ok;
                    tc_fence_after();
#pragma unroll
                    for (int c0 = 0; c0 < NH; c0 += 16) {
                        uint32_t v[16];
                        tmem_ld16(tcol + c0, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
                        tmem_wait_ld_regs<16>(v);
                        float h[16];
#pragma unroll
                        for (int u = 0; u < 16; ++u) h[u] = ok ? gam * __uint_as_float(v[u]) : 0.f;
                        tmem_st16(tcol + c0, reinterpret_cast<const uint32_t*>(h));
#pragma unroll
                        for (int i = 0; i < 16; i += 2) hp[(c0 + i) / 2] = pack_bf16(h[i], h[i + 1]);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(s_free);
                }
                mbar_arrive(&fac_empty[sl]);
                // (b) the next chunk's bf16 operand, as soon as DX and dB of this chunk have read
                // the current one (DX of the next chunk waits for it)
                if (more) {
                    wait_or_abort(g_free, it & 1, abort_flag, a.hdr);
                    write_g();
                }
                // (c) partial dB rows of this chunk -> staging -> reduce-add into the accumulator;
                // rows past the chunk's tokens add zero
                {
                    bool ok = wait_or_abort(db_full, it & 1, abort_flag, a.hdr);
                    tc_fence_after();
                    if (sct == 0) tma_store_wait_read<0>();  // previous reduce-add has read staging
                    named_sync(5, 256);
                    constexpr int HW = NH / 2;               // dB columns per lane half
                    constexpr int STEP = HW >= 32 ? 32 : 16;
                    const int nb0 = (wg - 2) * NH;
#pragma unroll
                    for (int c0 = 0; c0 < HW; c0 += STEP) {
                        uint32_t v[STEP];
                        tmem_ld16x2<HW>(tq + T_DB + nb0 + c0, &v[0]);
                        if constexpr (STEP == 32) tmem_ld16x2<HW>(tq + T_DB + nb0 + c0 + 16, &v[16]);
                        tmem_wait_ld_regs<STEP>(v);
                        const int n = nb0 + HW * hf + c0;
                        float val[STEP];
#pragma unroll
                        for (int u = 0; u < STEP; ++u)
                            val[u] = (ok && tt < vc) ? __uint_as_float(v[u]) : 0.f;
                        stage_row16(sm + Lay::OFF_DB, tt, n, val);
                        if constexpr (STEP == 32) stage_row16(sm + Lay::OFF_DB, tt, n + 16, val + 16);
                    }
                    tc_fence_before();
                    mbar_arrive(db_free);
                    fence_proxy_async();
                    named_sync(5, 256);
                    if (sct == 0) {
                        for (int j = 0; j < N / 32; ++j)
                            tma_reduce_add_3d(&map_acc, sm + Lay::OFF_DB + j * 8192, j * 32, g,
                                              (int)tok0);
                        tma_store_commit();
                    }
                }
            }
            if (sct == 0) tma_store_wait_all<0>();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

constexpr int state_smem_bytes(int N) {
    return kStateStages * StateSmem::stage_bytes(N) + (2 * kMaxSegChunks + 4) * 4 + 3 * kStateStages * 8 +
           8 + 16 + 1024;
}
// three CTAs of the aggregate kernel per SM (1 KB per CTA reserved by the system)
static_assert(3 * (state_smem_bytes(128) + 1024) <= 233472, "aggregate kernel occupancy");

template <typename K>
cudaError_t set_smem(K kernel, int bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <int N>
cudaError_t launch_l0(const Prob& pb, const Args& a, Launch& L, const CUtensorMap& mb,
                      const CUtensorMap& mc, bool write_tile = true) {
    const int cps = pb.Ls / kQ;
    const dim3 grid((unsigned)(pb.nseg_max * ((cps + kL0Chunks - 1) / kL0Chunks)), pb.G);
    cudaError_t e = set_smem(tc_l0_kernel<N>, l0_smem_bytes<N>());
    if (e != cudaSuccess) return e;
    L.begin("tc_l0");
    tc_l0_kernel<N><<<grid, kL0Threads, l0_smem_bytes<N>(), L.stream>>>(mb, mc, a,
                                                                        write_tile ? 1 : 0);
    return L.end();
}

cudaError_t launch_factors(const Prob& pb, const Args& a, Launch& L) {
    const int groups = (pb.Ls / kQ + kFacChunks - 1) / kFacChunks;
    const dim3 grid((unsigned)(pb.nseg_max * groups), (a.Hf + kFacHeads - 1) / kFacHeads);
    L.begin("tc_factors");
    tc_factors_kernel<<<grid, kFacThreads, 0, L.stream>>>(a);
    return L.end();
}

template <int N>
cudaError_t forward_n(const Prob& pb, const Args& a, Launch& L) {
    CUtensorMap mx, mb, mc;
    if (!make_map(&mx, a.x, pb.T, pb.H, kP) || !make_map(&mb, a.B, pb.T, pb.G, N) ||
        !make_map(&mc, a.C, pb.T, pb.G, N))
        return cudaErrorInvalidValue;
    cudaError_t e = launch_seg_table(pb, a, L);
    if (e != cudaSuccess) return e;
    if ((e = launch_l0<N>(pb, a, L, mb, mc)) != cudaSuccess) return e;
    if ((e = launch_factors(pb, a, L)) != cudaSuccess) return e;
    const dim3 grid((unsigned)(pb.nseg_max * a.npairs));
    e = set_smem(tc_seg_state_kernel<N, 0>, state_smem_bytes(N));
    if (e != cudaSuccess) return e;
    L.begin("tc_fwd_state");
    tc_seg_state_kernel<N, 0><<<grid, kStateThreads, state_smem_bytes(N), L.stream>>>(mx, mb, a);
    e = L.end();
    if (e != cudaSuccess) return e;
    e = launch_state_scan(pb, a, L, a.final_state != nullptr);
    if (e != cudaSuccess) return e;
    const long long items = pb.nseg_max * a.npairs;
    if constexpr (N == 64) {
        // persistent: two CTAs per SM, each walking items (segment, pair of heads)
        e = set_smem(tc_fwd_walk2_kernel, Walk2Layout::TOTAL);
        if (e != cudaSuccess) return e;
        const long long ctas = 2LL * sm_count();
        const dim3 pgrid((unsigned)(items < ctas ? items : ctas));
        L.begin("tc_fwd_walk");
        tc_fwd_walk2_kernel<<<pgrid, kWalk2Threads, Walk2Layout::TOTAL, L.stream>>>(mx, mb, mc, a);
    } else {
        // persistent: one CTA per SM, each walking items (segment, pair of heads)
        e = set_smem(tc_fwd_walk_kernel<N>, WalkLayout<N>::TOTAL);
        if (e != cudaSuccess) return e;
        const dim3 pgrid((unsigned)(items < sm_count() ? items : sm_count()));
        L.begin("tc_fwd_walk");
        tc_fwd_walk_kernel<N><<<pgrid, kWalkThreads, WalkLayout<N>::TOTAL, L.stream>>>(mx, mb, mc, a);
    }
    if ((e = L.end()) != cudaSuccess) return e;
    constexpr int fsmem = sizeof(float) * simt::walk_smem_floats(kP, N);
    L.begin("tc_fallback_walk");
    tc_fallback_walk_kernel<N><<<(unsigned)(2 * sm_count()), simt::kSimtThreads, fsmem, L.stream>>>(a);
    return L.end();
}

template <int N>
cudaError_t backward_n(const Prob& pb, const Args& a, Launch& L, bool reuse_forward) {
    CUtensorMap mx, mdy, mb, mc, mdb, mdc;
    if (!make_map(&mx, a.x, pb.T, pb.H, kP) || !make_map(&mdy, a.dy, pb.T, pb.H, kP) ||
        !make_map(&mb, a.B, pb.T, pb.G, N) || !make_map(&mc, a.C, pb.T, pb.G, N) ||
        !make_map_f32(&mdb, a.dbacc, pb.T, pb.G, N) || !make_map_f32(&mdc, a.dcacc, pb.T, pb.G, N))
        return cudaErrorInvalidValue;
    const dim3 grid((unsigned)(pb.nseg_max * a.npairs));
    cudaError_t e;
    if (reuse_forward) {
        // the forward's segment table, tiles, factors and segment states are in the
        // workspace; only check that they were made for these inputs, and add the fp32
        // C B^T tiles the forward does not make
        if ((e = launch_forward_match(pb, a, L)) != cudaSuccess) return e;
        if ((e = launch_l0<N>(pb, a, L, mb, mc, false)) != cudaSuccess) return e;
    } else {
        if ((e = launch_seg_table(pb, a, L)) != cudaSuccess) return e;
        if ((e = launch_l0<N>(pb, a, L, mb, mc)) != cudaSuccess) return e;
        if ((e = launch_factors(pb, a, L)) != cudaSuccess) return e;
        e = set_smem(tc_seg_state_kernel<N, 0>, state_smem_bytes(N));
        if (e != cudaSuccess) return e;
        L.begin("tc_fwd_state");
        tc_seg_state_kernel<N, 0><<<grid, kStateThreads, state_smem_bytes(N), L.stream>>>(mx, mb, a);
        if ((e = L.end()) != cudaSuccess) return e;
        if ((e = launch_state_scan(pb, a, L, false)) != cudaSuccess) return e;
    }
    e = set_smem(tc_seg_state_kernel<N, 1>, state_smem_bytes(N));
    if (e != cudaSuccess) return e;
    L.begin("tc_bwd_adj_state");
    tc_seg_state_kernel<N, 1><<<grid, kStateThreads, state_smem_bytes(N), L.stream>>>(mdy, mc, a);
    if ((e = L.end()) != cudaSuccess) return e;
    if ((e = launch_adjoint_scan(pb, a, L)) != cudaSuccess) return e;
    e = set_smem(tc_bwd_dc_kernel<N>, BwdLayout<N>::TOTAL);
    if (e != cudaSuccess) return e;
    L.begin("tc_bwd_dc");
    tc_bwd_dc_kernel<N><<<grid, kBwdThreads, BwdLayout<N>::TOTAL, L.stream>>>(mx, mdy, mb, mc, mdc,
                                                                             a);
    if ((e = L.end()) != cudaSuccess) return e;
    static_assert(DxLayout<N>::TOTAL <= 232448, "dx/dB walk shared memory");
    e = set_smem(tc_bwd_dxdb_kernel<N>, DxLayout<N>::TOTAL);
    if (e != cudaSuccess) return e;
    L.begin("tc_bwd_dxdb");
    tc_bwd_dxdb_kernel<N><<<grid, kDxThreads, DxLayout<N>::TOTAL, L.stream>>>(mx, mdy, mb, mc,
                                                                             mdb, a);
    if ((e = L.end()) != cudaSuccess) return e;
    return launch_dbc_convert(pb, a, L);
}

}  // namespace

bool tc_supported(int dtype, int P, int N, int Q, int H, int G) {
    (void)H;
    (void)G;
    return dtype == SSD_DTYPE_BF16 && P == kP && (N == 64 || N == 128) && Q == kQ &&
           encode_fn() != nullptr;
}

cudaError_t tc_forward(const Prob& pb, const Args& a, Launch& L) {
    return pb.N == 128 ? forward_n<128>(pb, a, L) : forward_n<64>(pb, a, L);
}

cudaError_t tc_backward(const Prob& pb, const Args& a, Launch& L, bool reuse_forward) {
    return pb.N == 128 ? backward_n<128>(pb, a, L, reuse_forward)
                       : backward_n<64>(pb, a, L, reuse_forward);
}

}  // namespace ssd
