// Internal declarations shared by the C-ABI layer and the kernel files.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ssd.h"

namespace ssd {

// One entry per segment: a run of whole chunks of one sequence.  Segments
// never straddle a sequence boundary, so the state only restarts at a
// segment's first token.
struct SegInfo {
    long long start;   // first token (packed index)
    int len;           // tokens in the segment (<= segment length)
    int seq;           // sequence (or dense row) index
    int flags;         // SEG_FIRST | SEG_LAST
    int pad[3];
};
static_assert(sizeof(SegInfo) == 32, "SegInfo layout");
enum { SEG_FIRST = 1, SEG_LAST = 2 };

// Header at the start of the workspace.
struct WsHeader {
    int status;   // first device-side error code (0 = none)
    int nseg;     // segments actually present
    // What the segment table was built for (written with it): the problem's sizes and
    // the input pointers.  ssd_backward_after_forward checks it before reusing the
    // forward's segment table, C B^T tiles, chunk factors and segment states.
    int sig_valid;
    int sig_dims[7];            // H, P, N, G, Ls, dtype, delta_init (bits)
    long long sig_T;
    const void* sig_ptr[6];     // x, raw_dt, B, C, cu_seqlens, initial_state
    int pad[40];
};
static_assert(sizeof(WsHeader) == 256, "WsHeader layout");

// A validated problem with derived sizes.
struct Prob {
    long long T;        // total tokens
    long long rowlen;   // tokens per dense row (0 for packed input)
    int nseq;           // sequences (dense rows or packed sequences)
    bool varlen;
    int H, P, N, G, Q;
    float delta_init;
    int dtype;
    int Ls;             // segment length in tokens (a multiple of Q)
    long long nseg_max; // upper bound on the number of segments
    bool tc;            // tensor-core path
};

// Byte offsets of the workspace regions.
struct Layout {
    size_t header, segtab, A, lam, scan_state, scan_dec, adj, rq, rqsuf, dbacc, dcacc, rtok, kfin, l0,
        fac, fb, cb32, total;
};

// Everything a kernel needs; passed by value.
struct Args {
    const void* x;
    const float* raw;
    const void* B;
    const void* C;
    const int* cu;
    const void* dy;
    void* y;
    float* final_state;
    const float* h0;   // [nseq][H][P][N] initial states (row-major), NULL: zero
    const float* dhT;  // [nseq][H][P][N] upstream gradient of final_state, NULL: zero
    float* dh0;        // [nseq][H][P][N] gradient of the initial states, NULL: not wanted
    void* dx;
    float* draw;
    void* dB;
    void* dC;
    WsHeader* hdr;
    SegInfo* segtab;
    float* A;       // [nseg_max][H][P][N]: segment aggregates, then the state entering each segment
    float* lam;     // [nseg_max][H]: segment log-decay, sum of -delta
    float* scan_state;  // [scan blocks][H][P][N]: block summaries of the scans over many segments
    float* scan_dec;    // [scan blocks][H]
    float* adj;     // [nseg_max][H][P][N]: adjoint aggregates, then the adjoint leaving each segment
    float* rq;      // [nseg_max][H]
    float* rqsuf;   // [nseg_max][H]
    float* dbacc;   // [T][G][N] fp32
    float* dcacc;   // [T][G][N] fp32
    float* kfin;    // [nseg_max][H]: <d final_state, final state> of a sequence's last segment
    float* rtok;    // [T][H] fp32 (tensor-core backward): the part of dy_t . y_t that comes from
                    // tokens before t's chunk
    unsigned char* l0;  // tensor-core path: [nseg_max][Ls / Q][G] 8 KB tiles, masked C B^T per chunk
    float* fac;         // tensor-core path: [nseg_max][Ls / Q][H] chunk factor records (kFacRec floats)
    int* fb;            // tensor-core path: [nseg_max][H / 2] 1 where a chunk of the (segment,
                        // head pair) has a delta sum beyond kMaxChunkDecay: that work item
                        // runs the SIMT evaluation instead
    float* cb32;        // tensor-core backward: [nseg_max][Ls / Q][G] lower triangles of the
                        // 64 x 64 fp32 C_t . B_s (s <= t), kCbTri floats each (cb_tri_row)
    long long T, rowlen;
    long long nseg_max;
    int nseq, H, P, N, G, Q, Ls;
    // Tensor-core work items take heads in pairs inside a B/C group: Hg = H / G heads per
    // group, ppg = (Hg + 1) / 2 pairs per group, npairs = G ppg.  With Hg odd, a group's
    // last pair has one head; its second slot is a dummy (zero x / dy tiles, zero factor
    // records, nothing written).  Factor records are kept per pair slot: Hf = 2 npairs
    // records per chunk (= H when Hg is even).
    int Hg, ppg, npairs, Hf;
    float delta_init;
    int dtype;
    int state_lm;   // A and adj stored lane-major (tensor-core path), see lm_row
};

// The heads of tensor-core pair p.
struct HeadPair {
    int h0;    // first head
    int g;     // B / C group
    bool v1;   // the second slot holds head h0 + 1
    int h1c;   // tile coordinate of the second slot: h0 + 1, or H (outside: zero tiles)
};
__host__ __device__ __forceinline__ HeadPair head_pair(const Args& a, int p) {
    HeadPair r;
    r.g = p / a.ppg;
    const int j = p - r.g * a.ppg;
    r.h0 = r.g * a.Hg + 2 * j;
    r.v1 = 2 * j + 1 < a.Hg;
    r.h1c = r.v1 ? r.h0 + 1 : a.H;
    return r;
}

// Segment states A / adj of one (segment, head) are P x N fp32.  The SIMT path keeps
// them row-major.  The tensor-core path keeps them lane-major: in each block of 32
// consecutive rows, columns 4k .. 4k+3 of row 32 b + l sit at float offset
// (32 k + l) * 4 of the block, so the 32 lanes of a warp, which hold 32 consecutive
// rows of a TMEM accumulator, move 512 contiguous bytes per float4.  lm_row gives
// float4 0 of row p; float4 k of the row is lm_row(..) + 128 k.
__host__ __device__ __forceinline__ long long lm_row(int p, int N) {
    return (long long)(p & ~31) * N + (p & 31) * 4;
}

// Packed lower triangle of a 64 x 64 tile: row t holds columns 0..t from float t (t + 1) / 2.
constexpr int kCbTri = 64 * 65 / 2;
__host__ __device__ __forceinline__ int cb_tri_row(int t) { return t * (t + 1) / 2; }

// Chunk factor record of one chunk and head (tensor-core path, chunk length 64):
// f[64], g[64], delta[64], half, then padding to a multiple of 16 bytes.
constexpr int kFacRec = 196;
enum { FAC_F = 0, FAC_G = 64, FAC_D = 128, FAC_HALF = 192 };

// Launch bookkeeping: counts kernels and, when profiling is on, brackets
// each launch with events on the launch stream.
struct Launch {
    cudaStream_t stream;
    int count = 0;
    void begin(const char* name);
    cudaError_t end();
};

// SIMT path (any supported shape, f32 or bf16).
cudaError_t simt_forward(const Prob& pb, const Args& a, Launch& L);
cudaError_t simt_backward(const Prob& pb, const Args& a, Launch& L);
// Tensor-core path (bf16, P = 64, N in {64, 128}, Q = 64, any number of heads per group).
cudaError_t tc_forward(const Prob& pb, const Args& a, Launch& L);
// reuse_forward: the workspace holds the forward's segment table, C B^T tiles, chunk
// factors and segment states for these inputs (checked on the device).
cudaError_t tc_backward(const Prob& pb, const Args& a, Launch& L, bool reuse_forward = false);
bool tc_supported(int dtype, int P, int N, int Q, int H, int G);

// SMs of the current device (persistent grids size themselves by it).
inline int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
        return 1;
    return n;
}

// One decode step for pb.nseq sequences (the batch rows).
cudaError_t launch_decode_step(const Prob& pb, const float* hin, float* hout, const void* x,
                               const float* raw, const void* B, const void* C, void* y,
                               cudaStream_t stream);

// Shared small kernels (segment table, state scans, gradient epilogues).
cudaError_t launch_seg_table(const Prob& pb, const Args& a, Launch& L);
// Checks that the workspace's segment table was built for this problem and these inputs;
// otherwise records SSD_ERR_WORKSPACE and empties the table, so that no kernel does work.
cudaError_t launch_forward_match(const Prob& pb, const Args& a, Launch& L);
// d_initial_state of the empty packed sequences: their d_final_state (or zero).
cudaError_t launch_empty_seq_grads(const Prob& pb, const Args& a, Launch& L);
// Blocks of segments the scans over segments summarise first (0: a single pass).
int scan_blocks(const Prob& pb);
cudaError_t launch_state_scan(const Prob& pb, const Args& a, Launch& L, bool write_final);
cudaError_t launch_adjoint_scan(const Prob& pb, const Args& a, Launch& L);
cudaError_t launch_bwd_epilogue(const Prob& pb, const Args& a, Launch& L);
cudaError_t launch_dbc_convert(const Prob& pb, const Args& a, Launch& L);

}  // namespace ssd
