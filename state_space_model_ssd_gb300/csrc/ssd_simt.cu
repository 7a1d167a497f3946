// SIMT path: every supported shape and dtype (fp32 problems always take it).
//
// Work unit = (segment, head); 256 threads; the P x N state lives in
// registers, thread (warp w, lane l) holding rows p = w + 8 r and columns
// n = l + 32 c.  Inside a segment the state advances token by token, i.e. the
// diagonal block of the semiseparable matrix (page "长序列 Mamba 多卡训练算力
// 和显存怎么同时省" §一) is evaluated as the recurrence itself, in fp32; only
// the segment aggregates cross between segments (ssd_scan.cu).
//
// Forward:  seg_state  A_j = sum_{t in j} exp(Lambda_end - Lambda_t) delta_t x_t B_t^T
//           state_scan H_in[j]
//           seg_walk   y_t = H_t C_t from H_in[j]
// Backward: seg_state + state_scan (recompute H_in), adj_state + adjoint_scan,
//           bwd_walk (dx, dB, dC, partial d_raw), epilogue (d_raw, dB/dC rounding).
//
// The delta gradient uses d delta_t = x_t.(G_t B_t) - sum_{u >= t} (r_u - q_u) with
// r_u = dy_u . y_u and q_u = delta_u x_u.(G_u B_u), which equals the direct
// reverse-mode expression <G_t, x_t B_t^T> - exp(-delta_t) <G_t, H_{t-1}>
// (both sides count the pairs s <= t <= u of the quadratic form).
#include "ssd_device.cuh"

namespace ssd {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int TT = 16;  // tokens staged in shared memory per step

template <typename TI>
__device__ __forceinline__ void load_rows(float* dst, const TI* src, long long tok0, int cnt,
                                          int H, int h, int width) {
    for (int i = threadIdx.x; i < cnt * width; i += kThreads) {
        const int j = i / width, k = i - j * width;
        dst[i] = ld_in(src, ((tok0 + j) * H + h) * (long long)width + k);
    }
}

__device__ __forceinline__ void load_deltas(float* ds, float* as, const float* raw,
                                            long long tok0, int cnt, int H, int h,
                                            float dinit) {
    for (int j = threadIdx.x; j < cnt; j += kThreads) {
        const float d = softplus_f(raw[(tok0 + j) * H + h] + dinit);
        ds[j] = d;
        as[j] = expf(-d);
    }
}

template <typename TI, int RP, int CP>
__global__ void __launch_bounds__(kThreads) simt_seg_state_kernel(Args a) {
    const int seg = blockIdx.x, h = blockIdx.y;
    if (seg >= a.hdr->nseg) return;
    const SegInfo si = a.segtab[seg];
    const int g = h / (a.H / a.G);
    const int P = a.P, N = a.N;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    extern __shared__ float sm[];
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
        load_rows(xs, X, tok0, cnt, a.H, h, P);
        load_rows(bs, Bm, tok0, cnt, a.G, g, N);
        load_deltas(ds, as, a.raw, tok0, cnt, a.H, h, a.delta_init);
        __syncthreads();
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
        __syncthreads();
    }
    float* A = a.A + ((long long)seg * a.H + h) * P * N;
#pragma unroll
    for (int r = 0; r < RP; ++r)
#pragma unroll
        for (int c = 0; c < CP; ++c) {
            const int n = lane + 32 * c;
            if (n < N) A[(warp + 8 * r) * N + n] = S[r][c];
        }
    if (threadIdx.x == 0) a.lam[(long long)seg * a.H + h] = lam;
}

template <typename TI, int RP, int CP>
__global__ void __launch_bounds__(kThreads) simt_seg_walk_kernel(Args a) {
    const int seg = blockIdx.x, h = blockIdx.y;
    if (seg >= a.hdr->nseg) return;
    const SegInfo si = a.segtab[seg];
    const int g = h / (a.H / a.G);
    const int P = a.P, N = a.N;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    extern __shared__ float sm[];
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
            S[r][c] = (n < N) ? Hin[(warp + 8 * r) * N + n] : 0.f;
        }
    for (int t0 = 0; t0 < si.len; t0 += TT) {
        const int cnt = min(TT, si.len - t0);
        const long long tok0 = si.start + t0;
        load_rows(xs, X, tok0, cnt, a.H, h, P);
        load_rows(bs, Bm, tok0, cnt, a.G, g, N);
        load_rows(cs, Cm, tok0, cnt, a.G, g, N);
        load_deltas(ds, as, a.raw, tok0, cnt, a.H, h, a.delta_init);
        __syncthreads();
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
        __syncthreads();
        for (int i = threadIdx.x; i < cnt * P; i += kThreads) {
            const int j = i / P, k = i - j * P;
            st_out(Y, ((tok0 + j) * a.H + h) * (long long)P + k, ys[i]);
        }
    }
}

// Adjoint aggregate of a segment: walking tokens backwards,
// G <- exp(-delta_t) (G + dy_t C_t^T); at the segment start G equals
// sum_u exp(Lambda_u - Lambda_before) dy_u C_u^T.
template <typename TI, int RP, int CP>
__global__ void __launch_bounds__(kThreads) simt_adj_state_kernel(Args a) {
    const int seg = blockIdx.x, h = blockIdx.y;
    if (seg >= a.hdr->nseg) return;
    const SegInfo si = a.segtab[seg];
    const int g = h / (a.H / a.G);
    const int P = a.P, N = a.N;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    extern __shared__ float sm[];
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
        load_rows(dys, DY, tok0, cnt, a.H, h, P);
        load_rows(cs, Cm, tok0, cnt, a.G, g, N);
        load_deltas(ds, as, a.raw, tok0, cnt, a.H, h, a.delta_init);
        __syncthreads();
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
        __syncthreads();
    }
    float* Ad = a.adj + ((long long)seg * a.H + h) * P * N;
#pragma unroll
    for (int r = 0; r < RP; ++r)
#pragma unroll
        for (int c = 0; c < CP; ++c) {
            const int n = lane + 32 * c;
            if (n < N) Ad[(warp + 8 * r) * N + n] = Gs[r][c];
        }
}

// Per (segment, head): forward sweep (state from H_in: dC and r = dy.y),
// then reverse sweep (adjoint from the scan: dx, dB, q and partial d_raw).
template <typename TI, int RP, int CP>
__global__ void __launch_bounds__(kThreads) simt_bwd_walk_kernel(Args a) {
    const int seg = blockIdx.x, h = blockIdx.y;
    if (seg >= a.hdr->nseg) return;
    const SegInfo si = a.segtab[seg];
    const int g = h / (a.H / a.G);
    const int P = a.P, N = a.N;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    extern __shared__ float sm[];
    float* xs = sm;
    float* bs = xs + TT * P;
    float* cs = bs + TT * N;
    float* dys = cs + TT * N;
    float* ds = dys + TT * P;
    float* as = ds + TT;
    float* red = as + TT;           // [kWarps][N]
    float* tmp = red + kWarps * N;  // [N]
    float* gbs = tmp + N;           // [P]
    float* xg = gbs + P;            // [P]
    float* rs = xg + P;             // [Ls]
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
                S[r][c] = (n < N) ? Hin[(warp + 8 * r) * N + n] : 0.f;
            }
    }
    // ---- forward sweep: dC_t += H_t^T dy_t, r_t = C_t . (H_t^T dy_t) = dy_t . y_t
    for (int t0 = 0; t0 < si.len; t0 += TT) {
        const int cnt = min(TT, si.len - t0);
        const long long tok0 = si.start + t0;
        load_rows(xs, X, tok0, cnt, a.H, h, P);
        load_rows(bs, Bm, tok0, cnt, a.G, g, N);
        load_rows(cs, Cm, tok0, cnt, a.G, g, N);
        load_rows(dys, DY, tok0, cnt, a.H, h, P);
        load_deltas(ds, as, a.raw, tok0, cnt, a.H, h, a.delta_init);
        __syncthreads();
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
            __syncthreads();
            for (int n = threadIdx.x; n < N; n += kThreads) {
                float v = 0.f;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) v += red[w * N + n];
                atomicAdd(a.dcacc + ((tok0 + j) * a.G + g) * (long long)N + n, v);
                tmp[n] = v * cs[j * N + n];
            }
            __syncthreads();
            if (warp == 0) {
                float v = 0.f;
                for (int n = lane; n < N; n += 32) v += tmp[n];
                v = warp_sum(v);
                if (lane == 0) rs[t0 + j] = v;
            }
        }
        __syncthreads();
    }
    // ---- reverse sweep from the adjoint arriving at the segment end
    float Gs[RP][CP];
    {
        const float* Gin = a.adj + ((long long)seg * a.H + h) * P * N;
#pragma unroll
        for (int r = 0; r < RP; ++r)
#pragma unroll
            for (int c = 0; c < CP; ++c) {
                const int n = lane + 32 * c;
                Gs[r][c] = (n < N) ? Gin[(warp + 8 * r) * N + n] : 0.f;
            }
    }
    float racc = 0.f;  // meaningful in thread 0 only
    const int ntiles = (si.len + TT - 1) / TT;
    for (int ti = ntiles - 1; ti >= 0; --ti) {
        const int t0 = ti * TT;
        const int cnt = min(TT, si.len - t0);
        const long long tok0 = si.start + t0;
        load_rows(xs, X, tok0, cnt, a.H, h, P);
        load_rows(bs, Bm, tok0, cnt, a.G, g, N);
        load_rows(cs, Cm, tok0, cnt, a.G, g, N);
        load_rows(dys, DY, tok0, cnt, a.H, h, P);
        load_deltas(ds, as, a.raw, tok0, cnt, a.H, h, a.delta_init);
        __syncthreads();
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
            __syncthreads();
            for (int p = threadIdx.x; p < P; p += kThreads) {
                const float gb = gbs[p];
                st_out(DX, ((tok0 + j) * a.H + h) * (long long)P + p, dt * gb);
                xg[p] = xs[j * P + p] * gb;
            }
            for (int n = threadIdx.x; n < N; n += kThreads) {
                float v = 0.f;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) v += red[w * N + n];
                atomicAdd(a.dbacc + ((tok0 + j) * a.G + g) * (long long)N + n, dt * v);
            }
            __syncthreads();
            if (warp == 0) {
                float v = 0.f;
                for (int p = lane; p < P; p += 32) v += xg[p];
                v = warp_sum(v);
                if (lane == 0) {
                    racc += rs[t0 + j] - dt * v;
                    a.draw[(tok0 + j) * a.H + h] = v - racc;
                }
            }
#pragma unroll
            for (int r = 0; r < RP; ++r)
#pragma unroll
                for (int c = 0; c < CP; ++c) Gs[r][c] *= at;
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) a.rq[(long long)seg * a.H + h] = racc;
}

template <typename K>
cudaError_t launch_kernel(K kernel, const char* name, const Prob& pb, const Args& a, Launch& L,
                          size_t smem) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)pb.nseg_max, pb.H);
    L.begin(name);
    kernel<<<grid, kThreads, smem, L.stream>>>(a);
    return L.end();
}

template <typename TI, int RP, int CP>
cudaError_t forward_impl(const Prob& pb, const Args& a, Launch& L) {
    const int P = pb.P, N = pb.N;
    cudaError_t e = launch_seg_table(pb, a, L);
    if (e != cudaSuccess) return e;
    e = launch_kernel(simt_seg_state_kernel<TI, RP, CP>, "simt_seg_state", pb, a, L,
                      sizeof(float) * (TT * P + TT * N + 2 * TT));
    if (e != cudaSuccess) return e;
    e = launch_state_scan(pb, a, L, a.final_state != nullptr);
    if (e != cudaSuccess) return e;
    return launch_kernel(simt_seg_walk_kernel<TI, RP, CP>, "simt_seg_walk", pb, a, L,
                         sizeof(float) * (2 * TT * P + 2 * TT * N + 2 * TT));
}

template <typename TI, int RP, int CP>
cudaError_t backward_impl(const Prob& pb, const Args& a, Launch& L) {
    const int P = pb.P, N = pb.N;
    cudaError_t e = launch_seg_table(pb, a, L);
    if (e != cudaSuccess) return e;
    e = launch_kernel(simt_seg_state_kernel<TI, RP, CP>, "simt_seg_state", pb, a, L,
                      sizeof(float) * (TT * P + TT * N + 2 * TT));
    if (e != cudaSuccess) return e;
    e = launch_state_scan(pb, a, L, false);
    if (e != cudaSuccess) return e;
    e = launch_kernel(simt_adj_state_kernel<TI, RP, CP>, "simt_adj_state", pb, a, L,
                      sizeof(float) * (TT * P + TT * N + 2 * TT));
    if (e != cudaSuccess) return e;
    e = launch_adjoint_scan(pb, a, L);
    if (e != cudaSuccess) return e;
    e = launch_kernel(simt_bwd_walk_kernel<TI, RP, CP>, "simt_bwd_walk", pb, a, L,
                      sizeof(float) * (2 * TT * P + 2 * TT * N + 2 * TT + kWarps * N + N +
                                       2 * P + pb.Ls));
    if (e != cudaSuccess) return e;
    return launch_bwd_epilogue(pb, a, L);
}

template <typename TI, int RP>
cudaError_t dispatch_cp(const Prob& pb, const Args& a, Launch& L, bool bwd) {
    switch ((pb.N + 31) / 32) {
        case 1: return bwd ? backward_impl<TI, RP, 1>(pb, a, L) : forward_impl<TI, RP, 1>(pb, a, L);
        case 2: return bwd ? backward_impl<TI, RP, 2>(pb, a, L) : forward_impl<TI, RP, 2>(pb, a, L);
        case 4: return bwd ? backward_impl<TI, RP, 4>(pb, a, L) : forward_impl<TI, RP, 4>(pb, a, L);
        default: return cudaErrorInvalidValue;
    }
}

template <typename TI>
cudaError_t dispatch(const Prob& pb, const Args& a, Launch& L, bool bwd) {
    switch (pb.P / 8) {
        case 1: return dispatch_cp<TI, 1>(pb, a, L, bwd);
        case 2: return dispatch_cp<TI, 2>(pb, a, L, bwd);
        case 4: return dispatch_cp<TI, 4>(pb, a, L, bwd);
        case 8: return dispatch_cp<TI, 8>(pb, a, L, bwd);
        case 16: return dispatch_cp<TI, 16>(pb, a, L, bwd);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t simt_forward(const Prob& pb, const Args& a, Launch& L) {
    return pb.dtype == SSD_DTYPE_BF16 ? dispatch<__nv_bfloat16>(pb, a, L, false)
                                      : dispatch<float>(pb, a, L, false);
}

cudaError_t simt_backward(const Prob& pb, const Args& a, Launch& L) {
    return pb.dtype == SSD_DTYPE_BF16 ? dispatch<__nv_bfloat16>(pb, a, L, true)
                                      : dispatch<float>(pb, a, L, true);
}

}  // namespace ssd
