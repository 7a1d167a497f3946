// The SIMT evaluation of one (segment, head): the recurrence itself, token by token, with
// the P x N state in registers (thread (warp w, lane l) holds rows p = w + 8 r and columns
// n = l + 32 c).  Inside a segment the diagonal block of the semiseparable matrix (page
// "长序列 Mamba 多卡训练算力和显存怎么同时省" §一) is evaluated as the recurrence, in fp32,
// which is exact for any delta; only segment states cross between segments (ssd_scan.cu).
//
// The bodies run on kSimtThreads threads of a block, which may be the whole block (the
// SIMT kernels) or its first kSimtThreads threads (the tensor-core kernels, for work items
// whose chunk decays leave the tensor-core factorisation's range); they synchronise with
// one named barrier.  States are read and written in the layout Args::state_lm names.
#pragma once

#include "ssd_device.cuh"

namespace ssd {
namespace simt {

constexpr int kSimtThreads = 256;
constexpr int kSimtWarps = kSimtThreads / 32;
constexpr int TT = 16;  // tokens staged in shared memory per step

struct Ctx {
    int tid;  // 0 .. kSimtThreads - 1
    int bar;  // named barrier id reserved for the body
    __device__ __forceinline__ void sync() const {
        asm volatile("bar.sync %0, %1;" ::"r"(bar), "n"(kSimtThreads) : "memory");
    }
};

// Offset of state element (p, n) of one (segment, head) block of P x N floats.
__device__ __forceinline__ long long st_idx(const Args& a, int p, int n) {
    return a.state_lm ? lm_row(p, a.N) + 128 * (n >> 2) + (n & 3) : (long long)p * a.N + n;
}

template <typename TI>
__device__ __forceinline__ void load_rows(const Ctx& cx, float* dst, const TI* src, long long tok0,
                                          int cnt, int H, int h, int width) {
    for (int i = cx.tid; i < cnt * width; i += kSimtThreads) {
        const int j = i / width, k = i - j * width;
        dst[i] = ld_in(src, ((tok0 + j) * H + h) * (long long)width + k);
    }
}

__device__ __forceinline__ void load_deltas(const Ctx& cx, float* ds, float* as, const float* raw,
                                            long long tok0, int cnt, int H, int h, float dinit) {
    for (int j = cx.tid; j < cnt; j += kSimtThreads) {
        const float d = softplus_f(raw[(tok0 + j) * H + h] + dinit);
        ds[j] = d;
        as[j] = expf(-d);
    }
}

// Shared memory (floats) each body needs.
__host__ __device__ constexpr int state_smem_floats(int P, int N) { return TT * P + TT * N + 2 * TT; }
__host__ __device__ constexpr int walk_smem_floats(int P, int N) {
    return 2 * TT * P + 2 * TT * N + 2 * TT;
}
__host__ __device__ constexpr int bwd_smem_floats(int P, int N, int Ls) {
    return 2 * TT * P + 2 * TT * N + 2 * TT + kSimtWarps * N + N + 2 * P + Ls + kSimtWarps;
}

// Segment aggregate A_j = sum_{t in j} exp(Lambda_end - Lambda_t) delta_t x_t B_t^T and the
// segment log-decay Lambda_end = -sum delta.
template <typename TI, int RP, int CP>
__device__ void seg_state_body(const Args& a, int seg, int h, float* sm, const Ctx& cx) {
    const SegInfo si = a.segtab[seg];
    const int g = h / (a.H / a.G);
    const int P = a.P, N = a.N;
    const int warp = cx.tid >> 5, lane = cx.tid & 31;
    float* xs = sm;
    float* bs = xs + TT * P;
    float* ds = bs + TT * N;
    float* as = ds + TT;
    const TI* X = static_cast<const TI*>(a.x);
    const TI* Bm = static_cast<const TI*>(a.B);
    float S[RP][CP];
#pragma unroll
    for (int r = 0; r < RP; ++r)
#pragma unroll
        for (int c = 0; c < CP; ++c) S[r][c] = 0.f;
    float lam = 0.f;
    for (int t0 = 0; t0 < si.len; t0 += TT) {
        const int cnt = min(TT, si.len - t0);
        const long long tok0 = si.start + t0;
        load_rows(cx, xs, X, tok0, cnt, a.H, h, P);
        load_rows(cx, bs, Bm, tok0, cnt, a.G, g, N);
        load_deltas(cx, ds, as, a.raw, tok0, cnt, a.H, h, a.delta_init);
        cx.sync();
        for (int j = 0; j < cnt; ++j) {
            const float at = as[j], dt = ds[j];
            lam -= dt;
#pragma unroll
            for (int r = 0; r < RP; ++r) {
                const float xv = dt * xs[j * P + warp + 8 * r];
#pragma unroll
                for (int c = 0; c < CP; ++c) {
                    const int n = lane + 32 * c;
                    const float bv = (n < N) ? bs[j * N + n] : 0.f;
                    S[r][c] = fmaf(at, S[r][c], xv * bv);
                }
            }
        }
        cx.sync();
    }
    float* A = a.A + ((long long)seg * a.H + h) * P * N;
#pragma unroll
    for (int r = 0; r < RP; ++r)
#pragma unroll
        for (int c = 0; c < CP; ++c) {
            const int n = lane + 32 * c;
            if (n < N) A[st_idx(a, warp + 8 * r, n)] = S[r][c];
        }
    if (cx.tid == 0) a.lam[(long long)seg * a.H + h] = lam;
}

// y_t = H_t C_t over the segment, from the state entering it.
template <typename TI, int RP, int CP>
__device__ void seg_walk_body(const Args& a, int seg, int h, float* sm, const Ctx& cx) {
    const SegInfo si = a.segtab[seg];
    const int g = h / (a.H / a.G);
    const int P = a.P, N = a.N;
    const int warp = cx.tid >> 5, lane = cx.tid & 31;
    float* xs = sm;
    float* bs = xs + TT * P;
    float* cs = bs + TT * N;
    float* ys = cs + TT * N;
    float* ds = ys + TT * P;
    float* as = ds + TT;
    const TI* X = static_cast<const TI*>(a.x);
    const TI* Bm = static_cast<const TI*>(a.B);
    const TI* Cm = static_cast<const TI*>(a.C);
    TI* Y = static_cast<TI*>(a.y);
    float S[RP][CP];
    const float* Hin = a.A + ((long long)seg * a.H + h) * P * N;
#pragma unroll
    for (int r = 0; r < RP; ++r)
#pragma unroll
        for (int c = 0; c < CP; ++c) {
            const int n = lane + 32 * c;
            S[r][c] = (n < N) ? Hin[st_idx(a, warp + 8 * r, n)] : 0.f;
        }
    for (int t0 = 0; t0 < si.len; t0 += TT) {
        const int cnt = min(TT, si.len - t0);
        const long long tok0 = si.start + t0;
        load_rows(cx, xs, X, tok0, cnt, a.H, h, P);
        load_rows(cx, bs, Bm, tok0, cnt, a.G, g, N);
        load_rows(cx, cs, Cm, tok0, cnt, a.G, g, N);
        load_deltas(cx, ds, as, a.raw, tok0, cnt, a.H, h, a.delta_init);
        cx.sync();
        for (int j = 0; j < cnt; ++j) {
            const float at = as[j], dt = ds[j];
#pragma unroll
            for (int r = 0; r < RP; ++r) {
                const float xv = dt * xs[j * P + warp + 8 * r];
                float yp = 0.f;
#pragma unroll
                for (int c = 0; c < CP; ++c) {
                    const int n = lane + 32 * c;
                    const bool ok = n < N;
                    const float bv = ok ? bs[j * N + n] : 0.f;
                    const float cv = ok ? cs[j * N + n] : 0.f;
                    S[r][c] = fmaf(at, S[r][c], xv * bv);
                    yp = fmaf(S[r][c], cv, yp);
                }
                yp = warp_sum(yp);
                if (lane == 0) ys[j * P + warp + 8 * r] = yp;
            }
        }
        cx.sync();
        for (int i = cx.tid; i < cnt * P; i += kSimtThreads) {
            const int j = i / P, k = i - j * P;
            st_out(Y, ((tok0 + j) * a.H + h) * (long long)P + k, ys[i]);
        }
    }
}

// Adjoint aggregate of a segment: walking tokens backwards,
// G <- exp(-delta_t) (G + dy_t C_t^T); at the segment start G equals
// sum_u exp(Lambda_u - Lambda_before) dy_u C_u^T.
template <typename TI, int RP, int CP>
__device__ void adj_state_body(const Args& a, int seg, int h, float* sm, const Ctx& cx) {
    const SegInfo si = a.segtab[seg];
    const int g = h / (a.H / a.G);
    const int P = a.P, N = a.N;
    const int warp = cx.tid >> 5, lane = cx.tid & 31;
    float* dys = sm;
    float* cs = dys + TT * P;
    float* ds = cs + TT * N;
    float* as = ds + TT;
    const TI* DY = static_cast<const TI*>(a.dy);
    const TI* Cm = static_cast<const TI*>(a.C);
    float Gs[RP][CP];
#pragma unroll
    for (int r = 0; r < RP; ++r)
#pragma unroll
        for (int c = 0; c < CP; ++c) Gs[r][c] = 0.f;
    const int ntiles = (si.len + TT - 1) / TT;
    for (int ti = ntiles - 1; ti >= 0; --ti) {
        const int t0 = ti * TT;
        const int cnt = min(TT, si.len - t0);
        const long long tok0 = si.start + t0;
        load_rows(cx, dys, DY, tok0, cnt, a.H, h, P);
        load_rows(cx, cs, Cm, tok0, cnt, a.G, g, N);
        load_deltas(cx, ds, as, a.raw, tok0, cnt, a.H, h, a.delta_init);
        cx.sync();
        for (int j = cnt - 1; j >= 0; --j) {
            const float at = as[j];
#pragma unroll
            for (int r = 0; r < RP; ++r) {
                const float dv = dys[j * P + warp + 8 * r];
#pragma unroll
                for (int c = 0; c < CP; ++c) {
                    const int n = lane + 32 * c;
                    const float cv = (n < N) ? cs[j * N + n] : 0.f;
                    Gs[r][c] = at * fmaf(dv, cv, Gs[r][c]);
                }
            }
        }
        cx.sync();
    }
    float* Ad = a.adj + ((long long)seg * a.H + h) * P * N;
#pragma unroll
    for (int r = 0; r < RP; ++r)
#pragma unroll
        for (int c = 0; c < CP; ++c) {
            const int n = lane + 32 * c;
            if (n < N) Ad[st_idx(a, warp + 8 * r, n)] = Gs[r][c];
        }
}

// Per (segment, head): forward sweep (state from H_in: dC and r = dy.y), then reverse
// sweep (adjoint from the scan: dx, dB, q and the delta gradient).  dB and dC are added
// into the fp32 accumulators.
//
// The delta gradient uses d delta_t = x_t.(G_t B_t) - sum_{u >= t} (r_u - q_u) with
// r_u = dy_u . y_u and q_u = delta_u x_u.(G_u B_u), which equals the direct reverse-mode
// expression <G_t, x_t B_t^T> - exp(-delta_t) <G_t, H_{t-1}> (both sides count the pairs
// s <= t <= u of the quadratic form).  The pairs beyond the segment end add
// <G_seg, H_end> (the adjoint arriving at the segment end and the state leaving it).
// finish = false leaves x.(G B) - sum_{u >= t in the segment} (r_u - q_u) in d_raw and
// the segment's sum of (r - q) in rq (ssd_scan.cu completes them); finish = true writes
// the finished d_raw_dt from the fp32 boundary term <G_seg, H_end> read from the scans'
// states.  Either way a sequence's last segment includes <d final_state, final state>.
template <typename TI, int RP, int CP>
__device__ void bwd_walk_body(const Args& a, int seg, int h, float* sm, const Ctx& cx,
                              bool finish) {
    const SegInfo si = a.segtab[seg];
    const int g = h / (a.H / a.G);
    const int P = a.P, N = a.N;
    const int warp = cx.tid >> 5, lane = cx.tid & 31;
    float* xs = sm;
    float* bs = xs + TT * P;
    float* cs = bs + TT * N;
    float* dys = cs + TT * N;
    float* ds = dys + TT * P;
    float* as = ds + TT;
    float* red = as + TT;               // [kSimtWarps][N]
    float* tmp = red + kSimtWarps * N;  // [N]
    float* gbs = tmp + N;               // [P]
    float* xg = gbs + P;                // [P]
    float* rs = xg + P;                 // [Ls]
    float* wred = rs + a.Ls;            // [kSimtWarps]
    const TI* X = static_cast<const TI*>(a.x);
    const TI* Bm = static_cast<const TI*>(a.B);
    const TI* Cm = static_cast<const TI*>(a.C);
    const TI* DY = static_cast<const TI*>(a.dy);
    TI* DX = static_cast<TI*>(a.dx);
    float S[RP][CP];
    {
        const float* Hin = a.A + ((long long)seg * a.H + h) * P * N;
#pragma unroll
        for (int r = 0; r < RP; ++r)
#pragma unroll
            for (int c = 0; c < CP; ++c) {
                const int n = lane + 32 * c;
                S[r][c] = (n < N) ? Hin[st_idx(a, warp + 8 * r, n)] : 0.f;
            }
    }
    // ---- forward sweep: dC_t += H_t^T dy_t, r_t = C_t . (H_t^T dy_t) = dy_t . y_t
    for (int t0 = 0; t0 < si.len; t0 += TT) {
        const int cnt = min(TT, si.len - t0);
        const long long tok0 = si.start + t0;
        load_rows(cx, xs, X, tok0, cnt, a.H, h, P);
        load_rows(cx, bs, Bm, tok0, cnt, a.G, g, N);
        load_rows(cx, cs, Cm, tok0, cnt, a.G, g, N);
        load_rows(cx, dys, DY, tok0, cnt, a.H, h, P);
        load_deltas(cx, ds, as, a.raw, tok0, cnt, a.H, h, a.delta_init);
        cx.sync();
        for (int j = 0; j < cnt; ++j) {
            const float at = as[j], dt = ds[j];
            float part[CP];
#pragma unroll
            for (int c = 0; c < CP; ++c) part[c] = 0.f;
#pragma unroll
            for (int r = 0; r < RP; ++r) {
                const int p = warp + 8 * r;
                const float xv = dt * xs[j * P + p];
                const float dv = dys[j * P + p];
#pragma unroll
                for (int c = 0; c < CP; ++c) {
                    const int n = lane + 32 * c;
                    const float bv = (n < N) ? bs[j * N + n] : 0.f;
                    S[r][c] = fmaf(at, S[r][c], xv * bv);
                    part[c] = fmaf(S[r][c], dv, part[c]);
                }
            }
#pragma unroll
            for (int c = 0; c < CP; ++c) {
                const int n = lane + 32 * c;
                if (n < N) red[warp * N + n] = part[c];
            }
            cx.sync();
            for (int n = cx.tid; n < N; n += kSimtThreads) {
                float v = 0.f;
#pragma unroll
                for (int w = 0; w < kSimtWarps; ++w) v += red[w * N + n];
                atomicAdd(a.dcacc + ((tok0 + j) * a.G + g) * (long long)N + n, v);
                tmp[n] = v * cs[j * N + n];
            }
            cx.sync();
            if (warp == 0) {
                float v = 0.f;
                for (int n = lane; n < N; n += 32) v += tmp[n];
                v = warp_sum(v);
                if (lane == 0) rs[t0 + j] = v;
            }
        }
        cx.sync();
    }
    // ---- reverse sweep from the adjoint arriving at the segment end
    float Gs[RP][CP];
    float kseg = 0.f;
    {
        const float* Gin = a.adj + ((long long)seg * a.H + h) * P * N;
        const float* Hend = a.A + ((long long)(seg + 1) * a.H + h) * P * N;
        const bool last = (si.flags & SEG_LAST) != 0;
        const bool more = finish && !last;
        // a sequence's last segment with an upstream final-state gradient: the pairs beyond
        // its end are <d final_state, final state>, and S holds the final state now
        const bool tail = last && a.dhT != nullptr;
        float kp = 0.f;
#pragma unroll
        for (int r = 0; r < RP; ++r)
#pragma unroll
            for (int c = 0; c < CP; ++c) {
                const int n = lane + 32 * c;
                Gs[r][c] = (n < N) ? Gin[st_idx(a, warp + 8 * r, n)] : 0.f;
                if (more && n < N) kp = fmaf(Gs[r][c], Hend[st_idx(a, warp + 8 * r, n)], kp);
                if (tail && n < N) kp = fmaf(Gs[r][c], S[r][c], kp);
            }
        if (finish || tail) {
            kp = warp_sum(kp);
            if (lane == 0) wred[warp] = kp;
            cx.sync();
#pragma unroll
            for (int w = 0; w < kSimtWarps; ++w) kseg += wred[w];
        }
    }
    float racc = 0.f;  // meaningful in thread 0 only
    const int ntiles = (si.len + TT - 1) / TT;
    for (int ti = ntiles - 1; ti >= 0; --ti) {
        const int t0 = ti * TT;
        const int cnt = min(TT, si.len - t0);
        const long long tok0 = si.start + t0;
        load_rows(cx, xs, X, tok0, cnt, a.H, h, P);
        load_rows(cx, bs, Bm, tok0, cnt, a.G, g, N);
        load_rows(cx, cs, Cm, tok0, cnt, a.G, g, N);
        load_rows(cx, dys, DY, tok0, cnt, a.H, h, P);
        load_deltas(cx, ds, as, a.raw, tok0, cnt, a.H, h, a.delta_init);
        cx.sync();
        for (int j = cnt - 1; j >= 0; --j) {
            const float at = as[j], dt = ds[j];
            float part[CP];
#pragma unroll
            for (int c = 0; c < CP; ++c) part[c] = 0.f;
#pragma unroll
            for (int r = 0; r < RP; ++r) {
                const int p = warp + 8 * r;
                const float dv = dys[j * P + p];
                const float xv = xs[j * P + p];
                float gb = 0.f;
#pragma unroll
                for (int c = 0; c < CP; ++c) {
                    const int n = lane + 32 * c;
                    const bool ok = n < N;
                    const float cv = ok ? cs[j * N + n] : 0.f;
                    const float bv = ok ? bs[j * N + n] : 0.f;
                    Gs[r][c] = fmaf(dv, cv, Gs[r][c]);
                    gb = fmaf(Gs[r][c], bv, gb);
                    part[c] = fmaf(Gs[r][c], xv, part[c]);
                }
                gb = warp_sum(gb);
                if (lane == 0) gbs[p] = gb;
            }
#pragma unroll
            for (int c = 0; c < CP; ++c) {
                const int n = lane + 32 * c;
                if (n < N) red[warp * N + n] = part[c];
            }
            cx.sync();
            for (int p = cx.tid; p < P; p += kSimtThreads) {
                const float gb = gbs[p];
                st_out(DX, ((tok0 + j) * a.H + h) * (long long)P + p, dt * gb);
                xg[p] = xs[j * P + p] * gb;
            }
            for (int n = cx.tid; n < N; n += kSimtThreads) {
                float v = 0.f;
#pragma unroll
                for (int w = 0; w < kSimtWarps; ++w) v += red[w * N + n];
                atomicAdd(a.dbacc + ((tok0 + j) * a.G + g) * (long long)N + n, dt * v);
            }
            cx.sync();
            if (warp == 0) {
                float v = 0.f;
                for (int p = lane; p < P; p += 32) v += xg[p];
                v = warp_sum(v);
                if (lane == 0) {
                    racc += rs[t0 + j] - dt * v;
                    const long long o = (tok0 + j) * a.H + h;
                    if (finish)
                        a.draw[o] = (v - racc - kseg) * sigmoid_f(a.raw[o] + a.delta_init);
                    else
                        a.draw[o] = v - racc - kseg;
                }
            }
#pragma unroll
            for (int r = 0; r < RP; ++r)
#pragma unroll
                for (int c = 0; c < CP; ++c) Gs[r][c] *= at;
        }
        cx.sync();
    }
    // the sum of (r - q) over the segment, and a last segment's final-state term, for the
    // earlier segments of the sequence
    if (!finish && cx.tid == 0) a.rq[(long long)seg * a.H + h] = racc + kseg;
}

}  // namespace simt
}  // namespace ssd
