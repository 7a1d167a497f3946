// Bidirectional mode (page "Mamba-2架构与LaCT并行计算技术解析" §3.1): the scan over the
// sequence and the scan over the flipped sequence, outputs concatenated along the last
// dimension.  Each sequence (dense row or packed sequence) is flipped on its own; the
// reverse direction's outputs are flipped back to the original token positions, so that
// y[t] = [y_forward[t] | y_reverse[t]], y_reverse[t] depending on tokens t .. end.
//
// The flipped copies of x, raw_dt, B, C and the two directions' outputs live in the
// caller's workspace; the passes themselves are ssd_forward / ssd_backward.
#include <string.h>

#include "ssd_device.cuh"

namespace ssd {
namespace {

// Token t's mirror inside its sequence: dense rows of rowlen tokens, or cu_seqlens.
struct Seqs {
    const int* cu;
    long long rowlen;
    __device__ __forceinline__ void bounds(int s, long long* b, long long* e) const {
        if (cu) {
            *b = cu[s];
            *e = cu[s + 1];
        } else {
            *b = (long long)s * rowlen;
            *e = *b + rowlen;
        }
    }
};

constexpr int kFlipThreads = 256;
constexpr int kFlipSplit = 64;  // CTAs per sequence (grid.y)

// dst[mirror(t)] = src[t] for rows of `words` 32-bit words (one row per token).
__global__ void __launch_bounds__(kFlipThreads)
    flip_rows_kernel(const uint32_t* src, uint32_t* dst, int words, Seqs q) {
    long long b, e;
    q.bounds(blockIdx.x, &b, &e);
    const long long n = (e - b) * words;
    for (long long i = (long long)blockIdx.y * blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.y * blockDim.x) {
        const long long t = i / words, w = i - t * words;
        dst[(e - 1 - t) * words + w] = src[(b + t) * words + w];
    }
}

// out[t][h] = [yf[t][h] | yr[mirror(t)][h]]: rows of hw words per direction and head.
__global__ void __launch_bounds__(kFlipThreads)
    concat_rows_kernel(const uint32_t* yf, const uint32_t* yr, uint32_t* out, int H, int hw,
                       Seqs q) {
    long long b, e;
    q.bounds(blockIdx.x, &b, &e);
    const long long per = (long long)H * 2 * hw;
    const long long n = (e - b) * per;
    for (long long i = (long long)blockIdx.y * blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.y * blockDim.x) {
        const long long t = b + i / per;
        const long long r = i - (t - b) * per;
        const int h = (int)(r / (2 * hw)), k = (int)(r - (long long)h * 2 * hw);
        out[t * per + r] = k < hw ? yf[(t * H + h) * hw + k]
                                  : yr[((e - 1 - (t - b)) * H + h) * hw + (k - hw)];
    }
}

// The upstream gradient of the concatenated output split by direction: df[t][h] its first
// half, dr[mirror(t)][h] its second half.
__global__ void __launch_bounds__(kFlipThreads)
    split_rows_kernel(const uint32_t* dy, uint32_t* df, uint32_t* dr, int H, int hw, Seqs q) {
    long long b, e;
    q.bounds(blockIdx.x, &b, &e);
    const long long per = (long long)H * 2 * hw;
    const long long n = (e - b) * per;
    for (long long i = (long long)blockIdx.y * blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.y * blockDim.x) {
        const long long t = b + i / per;
        const long long r = i - (t - b) * per;
        const int h = (int)(r / (2 * hw)), k = (int)(r - (long long)h * 2 * hw);
        if (k < hw)
            df[(t * H + h) * hw + k] = dy[t * per + r];
        else
            dr[((e - 1 - (t - b)) * H + h) * hw + (k - hw)] = dy[t * per + r];
    }
}

// acc[t] += src[mirror(t)] for rows of `n` elements (fp32 or bf16, summed in fp32).
template <typename T>
__global__ void __launch_bounds__(kFlipThreads)
    mirror_add_kernel(const T* src, T* acc, int n, Seqs q) {
    long long b, e;
    q.bounds(blockIdx.x, &b, &e);
    const long long total = (e - b) * n;
    for (long long i = (long long)blockIdx.y * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.y * blockDim.x) {
        const long long t = i / n, k = i - t * n;
        const long long d = (b + t) * n + k;
        st_out(acc, d, ld_in(acc, d) + ld_in(src, (e - 1 - t) * n + k));
    }
}

constexpr size_t kAlign = 256;
size_t up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// Workspace of the bidirectional calls: flipped x, raw_dt, B, C; the reverse direction's
// output and, in the backward, its upstream gradients and input gradients; then the
// single-direction workspace.
struct BiLayout {
    size_t xr, rawr, br, cr, yf, yr, dyf, dyr, dxr, drawr, dbr, dcr, inner, total;
};

BiLayout bi_layout(const ssd_problem_t* p, bool bwd, size_t inner_bytes) {
    const size_t T = (size_t)p->batch * p->seqlen;
    const size_t e = p->dtype == SSD_DTYPE_BF16 ? 2 : 4;
    const size_t xb = T * p->nheads * p->headdim * e, rb = T * p->nheads * 4,
                 bb = T * p->ngroups * p->dstate * e;
    BiLayout l;
    memset(&l, 0, sizeof(l));
    size_t off = 0;
    l.xr = off;
    off = up(off + xb);
    l.rawr = off;
    off = up(off + rb);
    l.br = off;
    off = up(off + bb);
    l.cr = off;
    off = up(off + bb);
    if (!bwd) {
        l.yf = off;
        off = up(off + xb);
        l.yr = off;
        off = up(off + xb);
    } else {
        l.dyf = off;
        off = up(off + xb);
        l.dyr = off;
        off = up(off + xb);
        l.dxr = off;
        off = up(off + xb);
        l.drawr = off;
        off = up(off + rb);
        l.dbr = off;
        off = up(off + bb);
        l.dcr = off;
        off = up(off + bb);
    }
    l.inner = off;
    l.total = off + inner_bytes;
    return l;
}

dim3 flip_grid(const ssd_problem_t* p) {
    return dim3((unsigned)(p->nseq > 0 ? p->nseq : p->batch), kFlipSplit);
}

cudaError_t flip(const void* src, void* dst, size_t row_bytes, const ssd_problem_t* p, Seqs q,
                 cudaStream_t s) {
    flip_rows_kernel<<<flip_grid(p), kFlipThreads, 0, s>>>(
        static_cast<const uint32_t*>(src), static_cast<uint32_t*>(dst), (int)(row_bytes / 4), q);
    return cudaGetLastError();
}

}  // namespace
}  // namespace ssd

using namespace ssd;

extern "C" {

ssd_status_t ssd_bidirectional_workspace_size(const ssd_problem_t* prob, int for_backward,
                                              size_t* bytes) {
    if (!bytes) return SSD_ERR_INVALID_ARG;
    size_t inner = 0;
    ssd_status_t st = ssd_workspace_size(prob, for_backward, &inner);
    if (st != SSD_OK) return st;
    *bytes = bi_layout(prob, for_backward != 0, inner).total;
    return SSD_OK;
}

ssd_status_t ssd_bidirectional_forward(const ssd_problem_t* prob, const void* x,
                                       const float* raw_dt, const void* B, const void* C,
                                       const int32_t* cu_seqlens, void* y,
                                       float* final_state_fwd, float* final_state_rev,
                                       void* workspace, size_t workspace_bytes, void* stream) {
    size_t inner = 0;
    ssd_status_t st = ssd_workspace_size(prob, 0, &inner);
    if (st != SSD_OK) return st;
    const BiLayout l = bi_layout(prob, false, inner);
    if (!workspace) return SSD_ERR_WORKSPACE;
    if ((uintptr_t)workspace % 256) return SSD_ERR_ALIGNMENT;
    if (workspace_bytes < l.total) return SSD_ERR_WORKSPACE;
    if ((prob->nseq > 0) != (cu_seqlens != nullptr)) return SSD_ERR_INVALID_ARG;
    const long long T = prob->batch * prob->seqlen;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* ws = static_cast<char*>(workspace);
    if (T > 0) {
        if (!x || !raw_dt || !B || !C || !y) return SSD_ERR_INVALID_ARG;
        if (((uintptr_t)x | (uintptr_t)raw_dt | (uintptr_t)B | (uintptr_t)C | (uintptr_t)y) & 15)
            return SSD_ERR_ALIGNMENT;
        const size_t e = prob->dtype == SSD_DTYPE_BF16 ? 2 : 4;
        const Seqs q{cu_seqlens, prob->nseq > 0 ? 0 : prob->seqlen};
        if (flip(x, ws + l.xr, (size_t)prob->nheads * prob->headdim * e, prob, q, s) != cudaSuccess ||
            flip(raw_dt, ws + l.rawr, (size_t)prob->nheads * 4, prob, q, s) != cudaSuccess ||
            flip(B, ws + l.br, (size_t)prob->ngroups * prob->dstate * e, prob, q, s) != cudaSuccess ||
            flip(C, ws + l.cr, (size_t)prob->ngroups * prob->dstate * e, prob, q, s) != cudaSuccess)
            return SSD_ERR_CUDA;
    }
    st = ssd_forward(prob, x, raw_dt, B, C, cu_seqlens, ws + l.yf, final_state_fwd, ws + l.inner,
                     inner, stream);
    if (st != SSD_OK) return st;
    st = ssd_forward(prob, ws + l.xr, reinterpret_cast<const float*>(ws + l.rawr), ws + l.br,
                     ws + l.cr, cu_seqlens, ws + l.yr, final_state_rev, ws + l.inner, inner,
                     stream);
    if (st != SSD_OK || T == 0) return st;
    const int hw = prob->headdim * (prob->dtype == SSD_DTYPE_BF16 ? 2 : 4) / 4;
    concat_rows_kernel<<<flip_grid(prob), kFlipThreads, 0, s>>>(
        reinterpret_cast<const uint32_t*>(ws + l.yf), reinterpret_cast<const uint32_t*>(ws + l.yr),
        static_cast<uint32_t*>(y), prob->nheads, hw,
        Seqs{cu_seqlens, prob->nseq > 0 ? 0 : prob->seqlen});
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

ssd_status_t ssd_bidirectional_backward(const ssd_problem_t* prob, const void* x,
                                        const float* raw_dt, const void* B, const void* C,
                                        const int32_t* cu_seqlens, const void* dy, void* dx,
                                        float* d_raw_dt, void* dB, void* dC, void* workspace,
                                        size_t workspace_bytes, void* stream) {
    size_t inner = 0;
    ssd_status_t st = ssd_workspace_size(prob, 1, &inner);
    if (st != SSD_OK) return st;
    const BiLayout l = bi_layout(prob, true, inner);
    if (!workspace) return SSD_ERR_WORKSPACE;
    if ((uintptr_t)workspace % 256) return SSD_ERR_ALIGNMENT;
    if (workspace_bytes < l.total) return SSD_ERR_WORKSPACE;
    if ((prob->nseq > 0) != (cu_seqlens != nullptr)) return SSD_ERR_INVALID_ARG;
    const long long T = prob->batch * prob->seqlen;
    if (T == 0) return SSD_OK;
    if (!x || !raw_dt || !B || !C || !dy || !dx || !d_raw_dt || !dB || !dC)
        return SSD_ERR_INVALID_ARG;
    if (((uintptr_t)x | (uintptr_t)raw_dt | (uintptr_t)B | (uintptr_t)C | (uintptr_t)dy |
         (uintptr_t)dx | (uintptr_t)d_raw_dt | (uintptr_t)dB | (uintptr_t)dC) & 15)
        return SSD_ERR_ALIGNMENT;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* ws = static_cast<char*>(workspace);
    const bool bf = prob->dtype == SSD_DTYPE_BF16;
    const size_t e = bf ? 2 : 4;
    const Seqs q{cu_seqlens, prob->nseq > 0 ? 0 : prob->seqlen};
    const size_t xrow = (size_t)prob->nheads * prob->headdim * e;
    const size_t brow = (size_t)prob->ngroups * prob->dstate * e;
    if (flip(x, ws + l.xr, xrow, prob, q, s) != cudaSuccess ||
        flip(raw_dt, ws + l.rawr, (size_t)prob->nheads * 4, prob, q, s) != cudaSuccess ||
        flip(B, ws + l.br, brow, prob, q, s) != cudaSuccess ||
        flip(C, ws + l.cr, brow, prob, q, s) != cudaSuccess)
        return SSD_ERR_CUDA;
    split_rows_kernel<<<flip_grid(prob), kFlipThreads, 0, s>>>(
        static_cast<const uint32_t*>(dy), reinterpret_cast<uint32_t*>(ws + l.dyf),
        reinterpret_cast<uint32_t*>(ws + l.dyr), prob->nheads, (int)(prob->headdim * e / 4), q);
    if (cudaGetLastError() != cudaSuccess) return SSD_ERR_CUDA;
    // forward direction straight into the outputs, the reverse one into the workspace
    st = ssd_backward(prob, x, raw_dt, B, C, cu_seqlens, ws + l.dyf, dx, d_raw_dt, dB, dC,
                      ws + l.inner, inner, stream);
    if (st != SSD_OK) return st;
    st = ssd_backward(prob, ws + l.xr, reinterpret_cast<const float*>(ws + l.rawr), ws + l.br,
                      ws + l.cr, cu_seqlens, ws + l.dyr, ws + l.dxr,
                      reinterpret_cast<float*>(ws + l.drawr), ws + l.dbr, ws + l.dcr,
                      ws + l.inner, inner, stream);
    if (st != SSD_OK) return st;
    // each input gradient adds the reverse direction's, flipped back
    const dim3 g = flip_grid(prob);
    const int nx = prob->nheads * prob->headdim, nb = prob->ngroups * prob->dstate;
    if (bf) {
        using B16 = __nv_bfloat16;
        mirror_add_kernel<B16><<<g, kFlipThreads, 0, s>>>(
            reinterpret_cast<const B16*>(ws + l.dxr), static_cast<B16*>(dx), nx, q);
        mirror_add_kernel<B16><<<g, kFlipThreads, 0, s>>>(
            reinterpret_cast<const B16*>(ws + l.dbr), static_cast<B16*>(dB), nb, q);
        mirror_add_kernel<B16><<<g, kFlipThreads, 0, s>>>(
            reinterpret_cast<const B16*>(ws + l.dcr), static_cast<B16*>(dC), nb, q);
    } else {
        mirror_add_kernel<float><<<g, kFlipThreads, 0, s>>>(
            reinterpret_cast<const float*>(ws + l.dxr), static_cast<float*>(dx), nx, q);
        mirror_add_kernel<float><<<g, kFlipThreads, 0, s>>>(
            reinterpret_cast<const float*>(ws + l.dbr), static_cast<float*>(dB), nb, q);
        mirror_add_kernel<float><<<g, kFlipThreads, 0, s>>>(
            reinterpret_cast<const float*>(ws + l.dcr), static_cast<float*>(dC), nb, q);
    }
    mirror_add_kernel<float><<<g, kFlipThreads, 0, s>>>(
        reinterpret_cast<const float*>(ws + l.drawr), d_raw_dt, prob->nheads, q);
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // extern "C"
