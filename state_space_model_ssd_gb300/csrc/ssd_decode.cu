// Single-token decode step: the recurrence of page "Mamba-2架构与LaCT并行计算技术解析"
// §1.1 advanced by one token for every sequence of a batch, from a carried state.
//
//   delta = softplus(raw_t + delta_init)
//   H     <- exp(-delta) H + delta x_t B_t^T        (H is P x N, fp32, read and written once)
//   y_t    = H C_t
//
// Bound by the state's bytes (2 P N 4 per sequence and head).  One CTA per (sequence,
// head); every thread moves float4 pieces of the state (16-byte loads and stores, each
// warp a contiguous 512-byte span), and the N / 4 threads of a state row reduce y_t[p]
// with shuffles.  The state may be updated in place (hin == hout): each piece is read,
// then written, by the same thread.
#include "ssd_device.cuh"

namespace ssd {

namespace {

constexpr int kDecThreads = 256;

template <typename TI>
__global__ void __launch_bounds__(kDecThreads)
    decode_step_kernel(const float* hin, float* hout, const TI* __restrict__ x,
                       const float* __restrict__ raw, const TI* __restrict__ Bm,
                       const TI* __restrict__ Cm, TI* y, int H, int P, int N, int G,
                       float delta_init) {
    __shared__ float xs[128], bs[128], cs[128];
    const int b = blockIdx.y, h = blockIdx.x, g = h / (H / G);
    const long long bh = (long long)b * H + h;
    const float delta = softplus_f(raw[bh] + delta_init);
    const float decay = expf(-delta);
    for (int i = threadIdx.x; i < P; i += blockDim.x) xs[i] = delta * ld_in(x, bh * P + i);
    for (int i = threadIdx.x; i < N; i += blockDim.x) {
        bs[i] = ld_in(Bm, ((long long)b * G + g) * N + i);
        cs[i] = ld_in(Cm, ((long long)b * G + g) * N + i);
    }
    __syncthreads();
    const int n4 = N >> 2;                       // float4 pieces per state row (2 .. 32)
    const int PN4 = P * n4;
    const float4* s4 = reinterpret_cast<const float4*>(hin + bh * P * N);
    float4* o4 = reinterpret_cast<float4*>(hout + bh * P * N);
    // every thread takes the same number of pieces, so the row reductions stay converged
    for (int e0 = 0; e0 < PN4; e0 += blockDim.x) {
        const int e = e0 + threadIdx.x;
        const bool in = e < PN4;
        const int p = e / n4, n = (e - p * n4) * 4;
        float part = 0.f;
        if (in) {
            const float4 v = s4[e];
            const float xv = xs[p];
            float4 w;
            w.x = fmaf(decay, v.x, xv * bs[n]);
            w.y = fmaf(decay, v.y, xv * bs[n + 1]);
            w.z = fmaf(decay, v.z, xv * bs[n + 2]);
            w.w = fmaf(decay, v.w, xv * bs[n + 3]);
            o4[e] = w;
            part = w.x * cs[n] + w.y * cs[n + 1] + w.z * cs[n + 2] + w.w * cs[n + 3];
        }
        // the n4 consecutive lanes of one row (n4 divides 32)
        for (int o = n4 >> 1; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o, n4);
        if (in && (e % n4) == 0) st_out(y, bh * P + p, part);
    }
}

}  // namespace

cudaError_t launch_decode_step(const Prob& pb, const float* hin, float* hout, const void* x,
                               const float* raw, const void* B, const void* C, void* y,
                               cudaStream_t stream) {
    const dim3 grid(pb.H, (unsigned)pb.nseq);
    if (pb.dtype == SSD_DTYPE_BF16)
        decode_step_kernel<__nv_bfloat16><<<grid, kDecThreads, 0, stream>>>(
            hin, hout, static_cast<const __nv_bfloat16*>(x), raw,
            static_cast<const __nv_bfloat16*>(B), static_cast<const __nv_bfloat16*>(C),
            static_cast<__nv_bfloat16*>(y), pb.H, pb.P, pb.N, pb.G, pb.delta_init);
    else
        decode_step_kernel<float><<<grid, kDecThreads, 0, stream>>>(
            hin, hout, static_cast<const float*>(x), raw, static_cast<const float*>(B),
            static_cast<const float*>(C), static_cast<float*>(y), pb.H, pb.P, pb.N, pb.G,
            pb.delta_init);
    return cudaGetLastError();
}

}  // namespace ssd
