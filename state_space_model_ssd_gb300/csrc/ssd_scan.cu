// Segment table, the state scans between segments, and the gradient
// epilogues.  These kernels are shared by the SIMT and tensor-core paths.
//
// The scan between segments is the one-GPU form of the state hand-off that
// page "揭秘MindSpeed-LLM多潜在注意力（MLA）与Mamba上下文并行实现原理" §三.2
// performs across devices (every part computes a local decay and a local
// state, then the prefix states are combined): here each segment contributes
// (decay_j, A_j) and the state entering segment j is
//     H_in[j] = decay_{j-1} * H_in[j-1] + A_{j-1},   H_in[first of a sequence] = 0,
// an associative combine (a1, S1) o (a2, S2) = (a1 a2, a2 S1 + S2).
#include "ssd_device.cuh"

namespace ssd {

namespace {

constexpr int kTableThreads = 1024;

// Builds the segment table from cu_seqlens (or the dense row length): every
// sequence is cut into segments of Ls tokens from its own start.  Checks the
// boundaries on the device and records SSD_ERR_DEVICE if they are malformed.
__device__ __forceinline__ void write_segment(const Args& a, long long base, int k, int cnt,
                                              long long start, int len, int s) {
    const long long idx = base + k;
    if (idx < a.nseg_max) {
        SegInfo e;
        e.start = start + (long long)k * a.Ls;
        e.len = min(a.Ls, len - k * a.Ls);
        e.seq = s;
        e.flags = (k == 0 ? SEG_FIRST : 0) | (k == cnt - 1 ? SEG_LAST : 0);
        e.pad[0] = e.pad[1] = e.pad[2] = 0;
        a.segtab[idx] = e;
    } else {
        set_status(a.hdr, SSD_ERR_DEVICE);
    }
}

// Sequences with more segments than this are written by the whole block.
constexpr int kOwnSegments = 8;

__global__ void __launch_bounds__(kTableThreads) seg_table_kernel(Args a) {
    __shared__ int warp_sums[32];
    __shared__ long long base_s;
    __shared__ int bad;
    __shared__ int nlong;
    __shared__ int long_seq[kTableThreads];
    __shared__ long long long_base[kTableThreads];
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    if (tid == 0) {
        // the pass starts here: no error yet, no table yet
        a.hdr->status = 0;
        a.hdr->sig_valid = 0;
        base_s = 0;
        bad = 0;
        if (a.cu && (a.cu[0] != 0 || (long long)a.cu[a.nseq] != a.T)) bad = 1;
    }
    __syncthreads();
    if (a.cu)
        for (int s = tid; s < a.nseq; s += blockDim.x)
            if (a.cu[s + 1] < a.cu[s]) bad = 1;
    __syncthreads();
    // final states that no segment writes: every row (zero) when the boundaries are
    // malformed, else the rows of empty packed sequences (their initial states, or zero)
    const long long row4 = (long long)a.H * a.P * a.N / 4;
    if (a.final_state && (bad || a.cu)) {
        float4* fs4 = reinterpret_cast<float4*>(a.final_state);
        const float4* h04 = reinterpret_cast<const float4*>(a.h0);
        // one sequence per thread and pass; the block writes the rows of the empty ones
        for (int s0 = 0; s0 < a.nseq; s0 += blockDim.x) {
            const int s = s0 + tid;
            const bool empty = s < a.nseq && (bad || a.cu[s + 1] == a.cu[s]);
            if (!__syncthreads_or(empty)) continue;
            for (int k = 0; k < (int)blockDim.x && s0 + k < a.nseq; ++k) {
                const int sk = s0 + k;
                if (bad || a.cu[sk + 1] == a.cu[sk])
                    for (long long i = tid; i < row4; i += blockDim.x)
                        fs4[(long long)sk * row4 + i] = (h04 && !bad)
                                                            ? h04[(long long)sk * row4 + i]
                                                            : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
    }
    if (bad) {
        if (tid == 0) {
            set_status(a.hdr, SSD_ERR_DEVICE);
            a.hdr->nseg = 0;
        }
        return;
    }
    // tensor-core path: no work item falls back to the SIMT evaluation until the chunk
    // factors say so
    if (a.fb)
        for (long long i = tid; i < a.nseg_max * a.npairs; i += blockDim.x) a.fb[i] = 0;
    for (int s0 = 0; s0 < a.nseq; s0 += blockDim.x) {
        const int s = s0 + tid;
        long long start = 0;
        int len = 0, cnt = 0;
        if (s < a.nseq) {
            start = a.cu ? (long long)a.cu[s] : (long long)s * a.rowlen;
            len = a.cu ? a.cu[s + 1] - a.cu[s] : (int)a.rowlen;
            cnt = (len + a.Ls - 1) / a.Ls;
        }
        int v = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += n;
        }
        if (lane == 31) warp_sums[w] = v;
        __syncthreads();
        if (w == 0) {
            int ws = (lane < (int)(blockDim.x >> 5)) ? warp_sums[lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, ws, o);
                if (lane >= o) ws += n;
            }
            warp_sums[lane] = ws;
        }
        __syncthreads();
        const int excl = v - cnt + (w > 0 ? warp_sums[w - 1] : 0);
        const long long base = base_s + excl;
        if (tid == 0) nlong = 0;
        __syncthreads();
        if (cnt <= kOwnSegments) {
            for (int k = 0; k < cnt; ++k) write_segment(a, base, k, cnt, start, len, s);
        } else {
            const int i = atomicAdd(&nlong, 1);
            long_seq[i] = s;
            long_base[i] = base;
        }
        __syncthreads();
        // the long sequences of this batch, one at a time, a segment per thread
        for (int i = 0; i < nlong; ++i) {
            const int sl = long_seq[i];
            const long long st = a.cu ? (long long)a.cu[sl] : (long long)sl * a.rowlen;
            const int ln = a.cu ? a.cu[sl + 1] - a.cu[sl] : (int)a.rowlen;
            const int cn = (ln + a.Ls - 1) / a.Ls;
            for (int k = tid; k < cn; k += blockDim.x)
                write_segment(a, long_base[i], k, cn, st, ln, sl);
        }
        __syncthreads();
        if (tid == (int)blockDim.x - 1) base_s += excl + cnt;
        __syncthreads();
    }
    if (tid == 0) {
        a.hdr->nseg = (int)(base_s < a.nseg_max ? base_s : a.nseg_max);
        WsHeader* h = a.hdr;
        h->sig_dims[0] = a.H;
        h->sig_dims[1] = a.P;
        h->sig_dims[2] = a.N;
        h->sig_dims[3] = a.G;
        h->sig_dims[4] = a.Ls;
        h->sig_dims[5] = a.dtype;
        h->sig_dims[6] = __float_as_int(a.delta_init);
        h->sig_T = a.T;
        h->sig_ptr[0] = a.x;
        h->sig_ptr[1] = a.raw;
        h->sig_ptr[2] = a.B;
        h->sig_ptr[3] = a.C;
        h->sig_ptr[4] = a.cu;
        h->sig_ptr[5] = a.h0;
        h->sig_valid = 1;
    }
}

// One thread: does the header describe a segment table built for this problem and these
// inputs?  If not, record SSD_ERR_WORKSPACE and empty the table.
__global__ void forward_match_kernel(Args a) {
    WsHeader* h = a.hdr;
    const bool ok = h->sig_valid == 1 && h->sig_T == a.T && h->sig_dims[0] == a.H &&
                    h->sig_dims[1] == a.P && h->sig_dims[2] == a.N && h->sig_dims[3] == a.G &&
                    h->sig_dims[4] == a.Ls && h->sig_dims[5] == a.dtype &&
                    h->sig_dims[6] == __float_as_int(a.delta_init) && h->sig_ptr[0] == a.x &&
                    h->sig_ptr[1] == a.raw && h->sig_ptr[2] == a.B && h->sig_ptr[3] == a.C &&
                    h->sig_ptr[4] == a.cu && h->sig_ptr[5] == a.h0;
    if (!ok) {
        set_status(h, SSD_ERR_WORKSPACE);
        h->nseg = 0;
    }
}

constexpr int kScanThreads = 128;
constexpr int kScanUnroll = 4;  // segments per batch; the next batch loads while this one is stored
// Scans over more than 2 kScanBlockSegs segments run in three passes: a summary of every
// block of kScanBlockSegs segments, a short serial pass over the block summaries, then
// each block's scan from its carry-in, so that the serial chain is kScanBlockSegs + blocks
// + kScanBlockSegs steps long instead of one step per segment.
constexpr int kScanBlockSegs = 64;

// Row-major float4 index of state piece e4 (final_state, the initial state and their
// gradients are row-major; the segment states may be lane-major).
__device__ __forceinline__ int row_major_e4(const Args& a, int e4) {
    if (!a.state_lm) return e4;
    const int N4 = a.N >> 2, blk = e4 / (32 * N4), j = e4 - blk * 32 * N4;
    return (blk * 32 + (j & 31)) * N4 + (j >> 5);
}

__device__ __forceinline__ float4 fma4(float d, float4 c, float4 g) {
    return make_float4(fmaf(d, c.x, g.x), fmaf(d, c.y, g.y), fmaf(d, c.z, g.z), fmaf(d, c.w, g.w));
}

// Forward scan over segments, per head and per state piece (4 elements per thread; the
// scan is the same for either storage order of the states).  On entry a.A holds the
// segment aggregates; on exit the state entering each segment (the sequence's initial
// state, or zero, at its first segment).  Optionally writes the state after the last
// segment of every sequence to final_state.
//   mode 0: every segment in one pass;
//   mode 1: the summary of block blockIdx.z: its carry-out from a zero carry-in and the
//           factor a carry-in gets by its end (zero once a sequence starts in the block);
//   mode 2: the scan of block blockIdx.z from its carry-in (bstate after the block pass).
__global__ void __launch_bounds__(kScanThreads)
    state_scan_kernel(Args a, int write_final, int mode, float4* bstate, float* bdec) {
    const int h = blockIdx.y;
    const int PN4 = (a.P * a.N) >> 2;
    const int e4 = blockIdx.x * blockDim.x + threadIdx.x;
    if (e4 >= PN4) return;
    const int nseg = a.hdr->nseg;
    const int blk = blockIdx.z;
    const int j0 = mode == 0 ? 0 : blk * kScanBlockSegs;
    const int j1 = mode == 0 ? nseg : min(nseg, j0 + kScanBlockSegs);
    const long long bi = ((long long)blk * a.H + h) * PN4 + e4;
    float4* A4 = reinterpret_cast<float4*>(a.A);
    const int fe4 = row_major_e4(a, e4);
    float4 carry = mode == 2 ? bstate[bi] : make_float4(0.f, 0.f, 0.f, 0.f);
    float dprod = 1.f;
    float4 agg[kScanUnroll], nagg[kScanUnroll];
    float dec[kScanUnroll], ndec[kScanUnroll];
    int flags[kScanUnroll], seq[kScanUnroll], nflags[kScanUnroll], nseqi[kScanUnroll];
    auto load = [&](int s0, float4* g, float* dc, int* fl, int* sq) {
#pragma unroll
        for (int u = 0; u < kScanUnroll; ++u) {
            const int s = s0 + u;
            if (s < j1) {
                g[u] = A4[((long long)s * a.H + h) * PN4 + e4];
                dc[u] = expf(a.lam[(long long)s * a.H + h]);
                fl[u] = a.segtab[s].flags;
                sq[u] = a.segtab[s].seq;
            }
        }
    };
    if (j0 < j1) load(j0, agg, dec, flags, seq);
    for (int s0 = j0; s0 < j1; s0 += kScanUnroll) {
        if (s0 + kScanUnroll < j1) load(s0 + kScanUnroll, nagg, ndec, nflags, nseqi);
#pragma unroll
        for (int u = 0; u < kScanUnroll; ++u) {
            const int s = s0 + u;
            if (s >= j1) break;
            if (flags[u] & SEG_FIRST) {
                carry = a.h0 ? reinterpret_cast<const float4*>(a.h0)[((long long)seq[u] * a.H + h) * PN4 + fe4]
                             : make_float4(0.f, 0.f, 0.f, 0.f);
                dprod = 0.f;
            }
            if (mode != 1) A4[((long long)s * a.H + h) * PN4 + e4] = carry;
            carry = fma4(dec[u], carry, agg[u]);
            dprod *= dec[u];
            if (mode != 1 && write_final && (flags[u] & SEG_LAST))
                reinterpret_cast<float4*>(a.final_state)[((long long)seq[u] * a.H + h) * PN4 + fe4] =
                    carry;
        }
#pragma unroll
        for (int u = 0; u < kScanUnroll; ++u) {
            agg[u] = nagg[u];
            dec[u] = ndec[u];
            flags[u] = nflags[u];
            seq[u] = nseqi[u];
        }
    }
    if (mode == 1) {
        bstate[bi] = carry;
        if (e4 == 0) bdec[(long long)blk * a.H + h] = dprod;
    }
}

// The serial pass over block summaries, per head and state piece: replaces each block's
// carry-out by its carry-in.  reverse: the adjoint's order (from the last block).
__global__ void __launch_bounds__(kScanThreads)
    scan_blocks_kernel(Args a, int nblk, int reverse, float4* bstate, const float* bdec) {
    const int h = blockIdx.y;
    const int PN4 = (a.P * a.N) >> 2;
    const int e4 = blockIdx.x * blockDim.x + threadIdx.x;
    if (e4 >= PN4) return;
    float4 c = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < nblk; ++k) {
        const int blk = reverse ? nblk - 1 - k : k;
        const long long bi = ((long long)blk * a.H + h) * PN4 + e4;
        const float4 out = bstate[bi];
        bstate[bi] = c;
        c = fma4(bdec[(long long)blk * a.H + h], c, out);
    }
}

// Reverse scan of the adjoint over segments.  On entry a.adj holds, per segment,
// sum_u exp(Lambda_u - Lambda_before) dy_u C_u^T; on exit the adjoint arriving at the
// segment's last token from later tokens of its sequence (the sequence's final-state
// gradient, or zero, at its last segment).  Writes d_initial_state (the adjoint before a
// sequence's first token) when asked.  Modes as state_scan_kernel's, blocks walked from
// their end.
__global__ void __launch_bounds__(kScanThreads)
    adjoint_scan_kernel(Args a, int mode, float4* bstate, float* bdec) {
    const int h = blockIdx.y;
    const int PN4 = (a.P * a.N) >> 2;
    const int e4 = blockIdx.x * blockDim.x + threadIdx.x;
    if (e4 >= PN4) return;
    const int nseg = a.hdr->nseg;
    const int blk = blockIdx.z;
    const int j0 = mode == 0 ? 0 : blk * kScanBlockSegs;
    const int j1 = mode == 0 ? nseg : min(nseg, j0 + kScanBlockSegs);
    const long long bi = ((long long)blk * a.H + h) * PN4 + e4;
    float4* G4 = reinterpret_cast<float4*>(a.adj);
    const int fe4 = row_major_e4(a, e4);
    float4 carry = mode == 2 ? bstate[bi] : make_float4(0.f, 0.f, 0.f, 0.f);
    float dprod = 1.f;
    float4 agg[kScanUnroll], nagg[kScanUnroll];
    float dec[kScanUnroll], ndec[kScanUnroll];
    int flags[kScanUnroll], nflags[kScanUnroll], seq[kScanUnroll], nseqi[kScanUnroll];
    auto load = [&](int s0, float4* g, float* dc, int* fl, int* sq) {
#pragma unroll
        for (int u = 0; u < kScanUnroll; ++u) {
            const int s = s0 - u;
            if (s >= j0) {
                g[u] = G4[((long long)s * a.H + h) * PN4 + e4];
                dc[u] = expf(a.lam[(long long)s * a.H + h]);
                fl[u] = a.segtab[s].flags;
                sq[u] = a.segtab[s].seq;
            }
        }
    };
    if (j0 < j1) load(j1 - 1, agg, dec, flags, seq);
    for (int s0 = j1 - 1; s0 >= j0; s0 -= kScanUnroll) {
        if (s0 - kScanUnroll >= j0) load(s0 - kScanUnroll, nagg, ndec, nflags, nseqi);
#pragma unroll
        for (int u = 0; u < kScanUnroll; ++u) {
            const int s = s0 - u;
            if (s < j0) break;
            const long long srow = ((long long)seq[u] * a.H + h) * PN4 + fe4;
            // the adjoint arriving at a sequence's last token: the gradient of its final state
            if (flags[u] & SEG_LAST) {
                carry = a.dhT ? reinterpret_cast<const float4*>(a.dhT)[srow]
                              : make_float4(0.f, 0.f, 0.f, 0.f);
                dprod = 0.f;
            }
            if (mode != 1) G4[((long long)s * a.H + h) * PN4 + e4] = carry;
            carry = fma4(dec[u], carry, agg[u]);
            dprod *= dec[u];
            // before a sequence's first token: the gradient of its initial state
            if (mode != 1 && a.dh0 && (flags[u] & SEG_FIRST))
                reinterpret_cast<float4*>(a.dh0)[srow] = carry;
        }
#pragma unroll
        for (int u = 0; u < kScanUnroll; ++u) {
            agg[u] = nagg[u];
            dec[u] = ndec[u];
            flags[u] = nflags[u];
            seq[u] = nseqi[u];
        }
    }
    if (mode == 1) {
        bstate[bi] = carry;
        if (e4 == 0) bdec[(long long)blk * a.H + h] = dprod;
    }
}

// d_initial_state of the empty packed sequences, which have no segment: their
// d_final_state (H = initial state at their end), or zero.
__global__ void empty_seq_grads_kernel(Args a) {
    const int s = blockIdx.x;
    if (a.cu[s + 1] != a.cu[s]) return;
    const long long row4 = (long long)a.H * a.P * a.N / 4;
    float4* d4 = reinterpret_cast<float4*>(a.dh0) + (long long)s * row4;
    const float4* t4 = reinterpret_cast<const float4*>(a.dhT) + (long long)s * row4;
    for (long long i = threadIdx.x; i < row4; i += blockDim.x)
        d4[i] = a.dhT ? t4[i] : make_float4(0.f, 0.f, 0.f, 0.f);
}

// Sum of (r - q) over the later segments of the same sequence, per head.
__global__ void rq_suffix_kernel(Args a) {
    const int h = blockIdx.x * blockDim.x + threadIdx.x;
    if (h >= a.H) return;
    const int nseg = a.hdr->nseg;
    float suf = 0.f;
    for (int s = nseg - 1; s >= 0; --s) {
        if (a.segtab[s].flags & SEG_LAST) suf = 0.f;
        a.rqsuf[(long long)s * a.H + h] = suf;
        suf += a.rq[(long long)s * a.H + h];
    }
}

// d_raw = (partial - later segments' sum of (r - q)) * sigmoid(raw + delta_init).
// On entry d_raw holds, per token, x.(G B) minus the in-segment suffix sum.
__global__ void ddt_finalize_kernel(Args a) {
    const int seg = blockIdx.x;
    if (seg >= a.hdr->nseg) return;
    const SegInfo si = a.segtab[seg];
    const long long base = si.start * a.H;
    const int cnt = si.len * a.H;
    for (int i = threadIdx.x; i < cnt; i += blockDim.x) {
        const int h = i % a.H;
        const float z = a.raw[base + i] + a.delta_init;
        a.draw[base + i] =
            (a.draw[base + i] - a.rqsuf[(long long)seg * a.H + h]) * sigmoid_f(z);
    }
}

// fp32 dB / dC accumulators -> outputs, four elements per thread and step (N is a
// multiple of 8, so T G N is a multiple of 4).
template <typename TO>
__global__ void dbc_convert_kernel(Args a) {
    const long long n4 = a.T * a.G * a.N / 4;
    TO* dB = static_cast<TO*>(a.dB);
    TO* dC = static_cast<TO*>(a.dC);
    const float4* b4 = reinterpret_cast<const float4*>(a.dbacc);
    const float4* c4 = reinterpret_cast<const float4*>(a.dcacc);
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4;
         i += (long long)gridDim.x * blockDim.x) {
        const float4 vb = b4[i], vc = c4[i];
        st_out4(dB, i, vb);
        st_out4(dC, i, vc);
    }
}

}  // namespace

cudaError_t launch_seg_table(const Prob& pb, const Args& a, Launch& L) {
    (void)pb;
    L.begin("seg_table");
    seg_table_kernel<<<1, kTableThreads, 0, L.stream>>>(a);
    return L.end();
}

cudaError_t launch_forward_match(const Prob& pb, const Args& a, Launch& L) {
    (void)pb;
    L.begin("forward_match");
    forward_match_kernel<<<1, 1, 0, L.stream>>>(a);
    return L.end();
}

cudaError_t launch_empty_seq_grads(const Prob& pb, const Args& a, Launch& L) {
    L.begin("empty_seq_grads");
    empty_seq_grads_kernel<<<(unsigned)pb.nseq, 256, 0, L.stream>>>(a);
    return L.end();
}

int scan_blocks(const Prob& pb) {
    return pb.nseg_max > 2 * kScanBlockSegs ? (int)((pb.nseg_max + kScanBlockSegs - 1) / kScanBlockSegs)
                                            : 0;
}

namespace {

template <typename K>
cudaError_t scan_three_pass(const Prob& pb, const Args& a, Launch& L, const char* name, K pass,
                            int reverse) {
    const int PN4 = (pb.P * pb.N) / 4;
    const int nblk = scan_blocks(pb);
    const dim3 g1((PN4 + kScanThreads - 1) / kScanThreads, pb.H, nblk);
    const dim3 g2((PN4 + kScanThreads - 1) / kScanThreads, pb.H);
    float4* bs = reinterpret_cast<float4*>(a.scan_state);
    L.begin(name);
    pass(g1, 1);
    cudaError_t e = L.end();
    if (e != cudaSuccess) return e;
    L.begin("scan_blocks");
    scan_blocks_kernel<<<g2, kScanThreads, 0, L.stream>>>(a, nblk, reverse, bs, a.scan_dec);
    if ((e = L.end()) != cudaSuccess) return e;
    L.begin(name);
    pass(g1, 2);
    return L.end();
}

}  // namespace

cudaError_t launch_state_scan(const Prob& pb, const Args& a, Launch& L, bool write_final) {
    const int PN4 = (pb.P * pb.N) / 4;
    float4* bs = reinterpret_cast<float4*>(a.scan_state);
    auto pass = [&](dim3 grid, int mode) {
        state_scan_kernel<<<grid, kScanThreads, 0, L.stream>>>(a, write_final ? 1 : 0, mode, bs,
                                                               a.scan_dec);
    };
    if (scan_blocks(pb)) return scan_three_pass(pb, a, L, "state_scan", pass, 0);
    L.begin("state_scan");
    pass(dim3((PN4 + kScanThreads - 1) / kScanThreads, pb.H), 0);
    return L.end();
}

cudaError_t launch_adjoint_scan(const Prob& pb, const Args& a, Launch& L) {
    const int PN4 = (pb.P * pb.N) / 4;
    float4* bs = reinterpret_cast<float4*>(a.scan_state);
    auto pass = [&](dim3 grid, int mode) {
        adjoint_scan_kernel<<<grid, kScanThreads, 0, L.stream>>>(a, mode, bs, a.scan_dec);
    };
    if (scan_blocks(pb)) return scan_three_pass(pb, a, L, "adjoint_scan", pass, 1);
    L.begin("adjoint_scan");
    pass(dim3((PN4 + kScanThreads - 1) / kScanThreads, pb.H), 0);
    return L.end();
}

cudaError_t launch_bwd_epilogue(const Prob& pb, const Args& a, Launch& L) {
    L.begin("rq_suffix");
    rq_suffix_kernel<<<(pb.H + 127) / 128, 128, 0, L.stream>>>(a);
    cudaError_t e = L.end();
    if (e != cudaSuccess) return e;
    L.begin("ddt_finalize");
    ddt_finalize_kernel<<<(unsigned)pb.nseg_max, 256, 0, L.stream>>>(a);
    e = L.end();
    if (e != cudaSuccess) return e;
    return launch_dbc_convert(pb, a, L);
}

cudaError_t launch_dbc_convert(const Prob& pb, const Args& a, Launch& L) {
    const long long n = pb.T * pb.G * pb.N / 4;
    long long blocks = (n + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    if (blocks < 1) blocks = 1;
    L.begin("dbc_convert");
    if (pb.dtype == SSD_DTYPE_BF16)
        dbc_convert_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, L.stream>>>(a);
    else
        dbc_convert_kernel<float><<<(unsigned)blocks, 256, 0, L.stream>>>(a);
    return L.end();
}

}  // namespace ssd
