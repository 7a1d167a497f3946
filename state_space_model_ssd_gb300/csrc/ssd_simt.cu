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
#include "simt_body.cuh"

namespace ssd {

namespace {

using simt::kSimtThreads;
constexpr int kThreads = kSimtThreads;

// One (segment, head) per block; the whole block runs the body.
template <typename TI, int RP, int CP>
__global__ void __launch_bounds__(kThreads) simt_seg_state_kernel(Args a) {
    if ((int)blockIdx.x >= a.hdr->nseg) return;
    extern __shared__ float sm[];
    simt::seg_state_body<TI, RP, CP>(a, blockIdx.x, blockIdx.y, sm, simt::Ctx{(int)threadIdx.x, 1});
}

template <typename TI, int RP, int CP>
__global__ void __launch_bounds__(kThreads) simt_seg_walk_kernel(Args a) {
    if ((int)blockIdx.x >= a.hdr->nseg) return;
    extern __shared__ float sm[];
    simt::seg_walk_body<TI, RP, CP>(a, blockIdx.x, blockIdx.y, sm, simt::Ctx{(int)threadIdx.x, 1});
}

template <typename TI, int RP, int CP>
__global__ void __launch_bounds__(kThreads) simt_adj_state_kernel(Args a) {
    if ((int)blockIdx.x >= a.hdr->nseg) return;
    extern __shared__ float sm[];
    simt::adj_state_body<TI, RP, CP>(a, blockIdx.x, blockIdx.y, sm, simt::Ctx{(int)threadIdx.x, 1});
}

template <typename TI, int RP, int CP>
__global__ void __launch_bounds__(kThreads) simt_bwd_walk_kernel(Args a) {
    if ((int)blockIdx.x >= a.hdr->nseg) return;
    extern __shared__ float sm[];
    simt::bwd_walk_body<TI, RP, CP>(a, blockIdx.x, blockIdx.y, sm,
                                    simt::Ctx{(int)threadIdx.x, 1}, false);
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
                      sizeof(float) * simt::state_smem_floats(P, N));
    if (e != cudaSuccess) return e;
    e = launch_state_scan(pb, a, L, a.final_state != nullptr);
    if (e != cudaSuccess) return e;
    return launch_kernel(simt_seg_walk_kernel<TI, RP, CP>, "simt_seg_walk", pb, a, L,
                         sizeof(float) * simt::walk_smem_floats(P, N));
}

template <typename TI, int RP, int CP>
cudaError_t backward_impl(const Prob& pb, const Args& a, Launch& L) {
    const int P = pb.P, N = pb.N;
    cudaError_t e = launch_seg_table(pb, a, L);
    if (e != cudaSuccess) return e;
    e = launch_kernel(simt_seg_state_kernel<TI, RP, CP>, "simt_seg_state", pb, a, L,
                      sizeof(float) * simt::state_smem_floats(P, N));
    if (e != cudaSuccess) return e;
    e = launch_state_scan(pb, a, L, false);
    if (e != cudaSuccess) return e;
    e = launch_kernel(simt_adj_state_kernel<TI, RP, CP>, "simt_adj_state", pb, a, L,
                      sizeof(float) * simt::state_smem_floats(P, N));
    if (e != cudaSuccess) return e;
    e = launch_adjoint_scan(pb, a, L);
    if (e != cudaSuccess) return e;
    e = launch_kernel(simt_bwd_walk_kernel<TI, RP, CP>, "simt_bwd_walk", pb, a, L,
                      sizeof(float) * simt::bwd_smem_floats(P, N, pb.Ls));
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
