// C ABI of the SSD scan library: argument checks, workspace layout, path
// dispatch and launch bookkeeping.  No kernel arithmetic lives here.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <functional>
#include <map>
#include <mutex>
#include <queue>
#include <string>
#include <tuple>
#include <vector>

#include "ssd_internal.cuh"

namespace ssd {

namespace {

thread_local int g_last_launches = 0;

// ---- profiler: events bracketing every launch while enabled
struct ProfRecord {
    std::string name;
    cudaEvent_t start, stop;
};
struct ProfTotal {
    std::string name;
    long long launches;
    double ms;
};
bool g_prof_on = false;
std::string g_prof_only;  // when not empty, only launches of this kernel are timed
std::vector<ProfRecord> g_prof_pending;
std::vector<ProfTotal> g_prof_totals;
std::vector<cudaEvent_t> g_event_pool;
const char* g_prof_name = nullptr;
cudaEvent_t g_prof_start = nullptr;

cudaEvent_t take_event() {
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

void prof_flush() {
    for (auto& r : g_prof_pending) {
        float ms = 0.f;
        cudaEventSynchronize(r.stop);
        cudaEventElapsedTime(&ms, r.start, r.stop);
        bool found = false;
        for (auto& t : g_prof_totals)
            if (t.name == r.name) {
                t.launches += 1;
                t.ms += ms;
                found = true;
                break;
            }
        if (!found) g_prof_totals.push_back({r.name, 1, (double)ms});
        g_event_pool.push_back(r.start);
        g_event_pool.push_back(r.stop);
    }
    g_prof_pending.clear();
}

constexpr size_t kAlign = 256;
size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool is_pow2_in(int v, int lo, int hi) {
    if (v < lo || v > hi) return false;
    return (v & (v - 1)) == 0;
}

// Segment length: whole chunks, and enough (segment, head) work units to
// fill the GPU several times over.  Up to 16 chunks as a rule; longer (up to 64)
// only while the units still fill the GPU 32 times, as on sequences of millions
// of tokens, where every segment boundary costs a materialised state read and
// written by each pass (64 x 64 x 4 bytes per head at N = 64 against 4096 tokens
// of x at 64 chunks).
int default_segment_chunks(long long T, int nseq, int H, int Q) {
    const long long target_units = 8LL * 152;
    const long long chunks = (T + Q - 1) / Q;
    const long long extra = nseq > 1 ? nseq : 0;
    int k = 16;
    while (k > 1 && (chunks / k + extra) * H < target_units) k >>= 1;
    if (k == 16)
        while (k < 64 && (chunks / (2 * k) + extra) * H >= 4 * target_units) k <<= 1;
    return k;
}

// Finishing time, in half-chunk steps, of a walk that runs one CTA per SM over the
// (segment, head pair) items of `rows` dense rows in launch order (the segments of each
// row in turn, head pairs fastest).  An item takes its chunk count plus a fixed start-up
// cost of about 2.5 chunks (state load, first tiles in flight, state store: measured on
// the backward walks) and goes to whichever of the `sms` SMs frees first.
long long walk_makespan(long long row_chunks, long long rows, int k, int npairs, int sms) {
    std::priority_queue<long long, std::vector<long long>, std::greater<long long>> free_at;
    for (int i = 0; i < sms; ++i) free_at.push(0);
    long long end = 0;
    const long long nseg = (row_chunks + k - 1) / k;
    for (long long r = 0; r < rows; ++r)
        for (long long s = 0; s < nseg; ++s) {
            const long long ch = s + 1 < nseg ? k : row_chunks - s * k;
            for (int p = 0; p < npairs; ++p) {
                const long long t = free_at.top() + 2 * ch + 5;
                free_at.pop();
                free_at.push(t);
                if (t > end) end = t;
            }
        }
    return end;
}

// Tensor-core path on dense rows, where the default rule gives 16 chunks: the walks
// are one CTA per SM over a few waves of work items, so the last wave's fill decides
// their time.  Of 8 to 64 chunks, the segment length with the shortest estimated
// walk (walk_makespan) wins, the longest of those within 1% of it (fewer segment
// boundaries).  Cached per shape.
int balanced_segment_chunks(long long row_chunks, long long rows, int npairs, int sms) {
    static std::mutex mu;
    static std::map<std::tuple<long long, long long, int, int>, int> cache;
    const auto key = std::make_tuple(row_chunks, rows, npairs, sms);
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    long long span[65] = {0};
    long long best = -1;
    for (int k = 8; k <= 64; ++k) {
        span[k] = walk_makespan(row_chunks, rows, k, npairs, sms);
        if (best < 0 || span[k] < best) best = span[k];
    }
    int pick = 16;
    for (int k = 8; k <= 64; ++k)
        if (span[k] * 100 <= best * 101) pick = k;
    std::lock_guard<std::mutex> lock(mu);
    cache[key] = pick;
    return pick;
}

int choose_segment_length(const Prob& b) {
    // SSD_SEGMENT_CHUNKS (1..64) fixes the number of chunks per segment; the
    // result does not depend on it (tests use it to cover multi-chunk segments
    // at small sizes).
    if (const char* env = getenv("SSD_SEGMENT_CHUNKS")) {
        const int k = atoi(env);
        if (k >= 1 && k <= 64) return k * b.Q;
    }
    const int k = default_segment_chunks(b.T, b.nseq, b.H, b.Q);
    if (k != 16 || !b.tc || b.varlen) return k * b.Q;
    const int sms = sm_count();
    const long long row_chunks = (b.rowlen + b.Q - 1) / b.Q;
    const int npairs = b.G * ((b.H / b.G + 1) / 2);
    // no device to size for, or a simulation too long to run on the host
    if (sms < 8 || row_chunks * b.nseq * npairs > (1LL << 20)) return k * b.Q;
    return balanced_segment_chunks(row_chunks, b.nseq, npairs, sms) * b.Q;
}

ssd_status_t make_prob(const ssd_problem_t* p, Prob* out) {
    if (!p || !out) return SSD_ERR_INVALID_ARG;
    if (p->batch < 1 || p->seqlen < 0 || p->nheads < 1 || p->ngroups < 1 || p->nseq < 0)
        return SSD_ERR_INVALID_ARG;
    if (p->nheads % p->ngroups != 0) return SSD_ERR_INVALID_ARG;
    if (!isfinite(p->delta_init)) return SSD_ERR_INVALID_ARG;
    if (p->dtype != SSD_DTYPE_F32 && p->dtype != SSD_DTYPE_BF16) return SSD_ERR_INVALID_ARG;
    if (p->headdim < 1 || p->dstate < 1 || p->chunk_size < 1) return SSD_ERR_INVALID_ARG;
    if (p->nseq > 0 && p->batch != 1) return SSD_ERR_INVALID_ARG;
    if (!is_pow2_in(p->headdim, 8, 128) || !is_pow2_in(p->dstate, 8, 128) ||
        !is_pow2_in(p->chunk_size, 16, 256))
        return SSD_ERR_UNSUPPORTED;
    const long long T = p->batch * p->seqlen;
    if (p->seqlen > 0x7fffffffLL || T > 0x7fffffffLL) return SSD_ERR_UNSUPPORTED;
    Prob& b = *out;
    b.T = T;
    b.varlen = p->nseq > 0;
    b.nseq = b.varlen ? p->nseq : (int)p->batch;
    b.rowlen = b.varlen ? 0 : p->seqlen;
    b.H = p->nheads;
    b.P = p->headdim;
    b.N = p->dstate;
    b.G = p->ngroups;
    b.Q = p->chunk_size;
    b.delta_init = p->delta_init;
    b.dtype = p->dtype;
    // Fewer tokens than one chunk: the tensor-core tiles would be mostly padding, and the
    // SIMT path's fp32 products keep a lone token's head-summed dB / dC exact where the
    // heads' terms cancel (bf16 operands would leave their rounding in the small sum).
    b.tc = T >= p->chunk_size &&
           tc_supported(p->dtype, p->headdim, p->dstate, p->chunk_size, p->nheads, p->ngroups);
    b.Ls = choose_segment_length(b);
    // every sequence (dense row) may end in a partial segment
    b.nseg_max = (T + b.Ls - 1) / b.Ls + b.nseq;
    if (b.nseg_max < 1) b.nseg_max = 1;
    if (b.nseg_max > 0x7fffffffLL) return SSD_ERR_UNSUPPORTED;
    return SSD_OK;
}

Layout make_layout(const Prob& b, bool bwd) {
    Layout l;
    size_t off = 0;
    const size_t PN = (size_t)b.P * b.N;
    l.header = off;
    off = align_up(off + sizeof(WsHeader));
    l.segtab = off;
    off = align_up(off + sizeof(SegInfo) * (size_t)b.nseg_max);
    l.A = off;
    off = align_up(off + sizeof(float) * (size_t)b.nseg_max * b.H * PN);
    l.lam = off;
    off = align_up(off + sizeof(float) * (size_t)b.nseg_max * b.H);
    l.scan_state = l.scan_dec = 0;
    if (const int nblk = scan_blocks(b)) {
        l.scan_state = off;
        off = align_up(off + sizeof(float) * (size_t)nblk * b.H * PN);
        l.scan_dec = off;
        off = align_up(off + sizeof(float) * (size_t)nblk * b.H);
    }
    // regions both passes use come first, so that a forward's workspace is a prefix of
    // the backward's (ssd_backward_after_forward reuses it)
    l.l0 = l.fac = l.fb = 0;
    if (b.tc) {  // one 64 x 64 bf16 tile per chunk slot of every segment and group
        l.l0 = off;
        off = align_up(off + (size_t)8192 * b.nseg_max * (b.Ls / b.Q) * b.G);
        // one factor record per chunk slot and head slot of every pair
        const int npairs = b.G * ((b.H / b.G + 1) / 2);
        l.fac = off;
        off = align_up(off + sizeof(float) * kFacRec * b.nseg_max * (b.Ls / b.Q) * 2 * npairs);
        // one fallback flag per (segment, head pair)
        l.fb = off;
        off = align_up(off + sizeof(int) * b.nseg_max * npairs);
    }
    l.adj = l.rq = l.rqsuf = l.dbacc = l.dcacc = l.rtok = l.kfin = l.cb32 = 0;
    if (bwd) {
        l.kfin = off;
        off = align_up(off + sizeof(float) * (size_t)b.nseg_max * b.H);
        l.adj = off;
        off = align_up(off + sizeof(float) * (size_t)b.nseg_max * b.H * PN);
        l.rq = off;
        off = align_up(off + sizeof(float) * (size_t)b.nseg_max * b.H);
        l.rqsuf = off;
        off = align_up(off + sizeof(float) * (size_t)b.nseg_max * b.H);
        l.dbacc = off;
        off = align_up(off + sizeof(float) * (size_t)b.T * b.G * b.N);
        l.dcacc = off;
        off = align_up(off + sizeof(float) * (size_t)b.T * b.G * b.N);
        l.rtok = off;
        off = align_up(off + sizeof(float) * (size_t)b.T * b.H);
        if (b.tc) {  // fp32 C B^T lower triangle per chunk slot of every segment and group
            l.cb32 = off;
            off = align_up(off + sizeof(float) * kCbTri * b.nseg_max * (b.Ls / b.Q) * b.G);
        }
    }
    l.total = off;
    return l;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

Args make_args(const Prob& b, const Layout& l, void* ws) {
    Args a;
    memset(&a, 0, sizeof(a));
    char* base = static_cast<char*>(ws);
    a.hdr = reinterpret_cast<WsHeader*>(base + l.header);
    a.segtab = reinterpret_cast<SegInfo*>(base + l.segtab);
    a.A = reinterpret_cast<float*>(base + l.A);
    a.lam = reinterpret_cast<float*>(base + l.lam);
    if (l.scan_state) {
        a.scan_state = reinterpret_cast<float*>(base + l.scan_state);
        a.scan_dec = reinterpret_cast<float*>(base + l.scan_dec);
    }
    if (l.adj) {
        a.adj = reinterpret_cast<float*>(base + l.adj);
        a.rq = reinterpret_cast<float*>(base + l.rq);
        a.rqsuf = reinterpret_cast<float*>(base + l.rqsuf);
        a.dbacc = reinterpret_cast<float*>(base + l.dbacc);
        a.dcacc = reinterpret_cast<float*>(base + l.dcacc);
        a.rtok = reinterpret_cast<float*>(base + l.rtok);
        a.kfin = reinterpret_cast<float*>(base + l.kfin);
    }
    if (l.l0) a.l0 = reinterpret_cast<unsigned char*>(base + l.l0);
    if (l.fac) a.fac = reinterpret_cast<float*>(base + l.fac);
    if (l.fb) a.fb = reinterpret_cast<int*>(base + l.fb);
    if (l.cb32) a.cb32 = reinterpret_cast<float*>(base + l.cb32);
    a.T = b.T;
    a.rowlen = b.rowlen;
    a.nseg_max = b.nseg_max;
    a.nseq = b.nseq;
    a.H = b.H;
    a.P = b.P;
    a.N = b.N;
    a.G = b.G;
    a.Hg = b.H / b.G;
    a.ppg = (a.Hg + 1) / 2;
    a.npairs = b.G * a.ppg;
    a.Hf = 2 * a.npairs;
    a.Q = b.Q;
    a.Ls = b.Ls;
    a.delta_init = b.delta_init;
    a.dtype = b.dtype;
    a.state_lm = l.l0 ? 1 : 0;
    return a;
}

ssd_status_t check_common(const ssd_problem_t* prob, const int32_t* cu, void* ws,
                          size_t ws_bytes, bool bwd, Prob* b, Layout* l) {
    ssd_status_t st = make_prob(prob, b);
    if (st != SSD_OK) return st;
    if ((prob->nseq > 0) != (cu != nullptr)) return SSD_ERR_INVALID_ARG;
    if (cu && ((uintptr_t)cu & 3u)) return SSD_ERR_ALIGNMENT;
    *l = make_layout(*b, bwd);
    if (!ws) return SSD_ERR_WORKSPACE;
    if ((uintptr_t)ws % kAlign) return SSD_ERR_ALIGNMENT;
    if (ws_bytes < l->total) return SSD_ERR_WORKSPACE;
    return SSD_OK;
}

}  // namespace

void Launch::begin(const char* name) {
    ++count;
    if (g_prof_on && (g_prof_only.empty() || g_prof_only == name)) {
        g_prof_name = name;
        g_prof_start = take_event();
        if (g_prof_start) cudaEventRecord(g_prof_start, stream);
    }
}

cudaError_t Launch::end() {
    cudaError_t e = cudaGetLastError();
    if (g_prof_on && g_prof_start) {
        cudaEvent_t stop = take_event();
        if (stop) {
            cudaEventRecord(stop, stream);
            g_prof_pending.push_back({std::string(g_prof_name), g_prof_start, stop});
        }
        g_prof_start = nullptr;
    }
    return e;
}

}  // namespace ssd

using namespace ssd;

extern "C" {

int ssd_version(void) { return SSD_API_VERSION; }

const char* ssd_status_string(ssd_status_t s) {
    switch (s) {
        case SSD_OK: return "ok";
        case SSD_ERR_INVALID_ARG: return "invalid argument";
        case SSD_ERR_UNSUPPORTED: return "unsupported problem shape";
        case SSD_ERR_ALIGNMENT: return "misaligned pointer";
        case SSD_ERR_WORKSPACE:
            return "workspace missing or too small, or not holding the matching forward";
        case SSD_ERR_CUDA: return "CUDA runtime error";
        case SSD_ERR_TIMEOUT: return "device-side wait timed out";
        case SSD_ERR_DEVICE: return "device-side check failed";
    }
    return "unknown status";
}

ssd_status_t ssd_workspace_size(const ssd_problem_t* prob, int for_backward, size_t* bytes) {
    if (!bytes) return SSD_ERR_INVALID_ARG;
    Prob b;
    ssd_status_t st = make_prob(prob, &b);
    if (st != SSD_OK) return st;
    *bytes = make_layout(b, for_backward != 0).total;
    return SSD_OK;
}

const char* ssd_dispatch_path(const ssd_problem_t* prob, int for_backward) {
    (void)for_backward;
    Prob b;
    if (make_prob(prob, &b) != SSD_OK) return nullptr;
    return b.tc ? "tensor-core" : "simt";
}

int ssd_last_launch_count(void) { return g_last_launches; }

ssd_status_t ssd_forward_state(const ssd_problem_t* prob, const void* x, const float* raw_dt,
                               const void* B, const void* C, const int32_t* cu_seqlens,
                               const float* initial_state, void* y, float* final_state,
                               void* workspace, size_t workspace_bytes, void* stream) {
    g_last_launches = 0;
    Prob b;
    Layout l;
    ssd_status_t st = check_common(prob, cu_seqlens, workspace, workspace_bytes, false, &b, &l);
    if (st != SSD_OK) return st;
    if (initial_state && !aligned16(initial_state)) return SSD_ERR_ALIGNMENT;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t sbytes = sizeof(float) * (size_t)b.nseq * b.H * b.P * b.N;
    if (b.T == 0) {  // nothing to read: the final states are the initial ones (or zero)
        if (final_state) {
            const cudaError_t e =
                initial_state ? cudaMemcpyAsync(final_state, initial_state, sbytes,
                                                cudaMemcpyDeviceToDevice, s)
                              : cudaMemsetAsync(final_state, 0, sbytes, s);
            if (e != cudaSuccess) return SSD_ERR_CUDA;
        }
        return SSD_OK;
    }
    if (!x || !raw_dt || !B || !C || !y) return SSD_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(raw_dt) || !aligned16(B) || !aligned16(C) || !aligned16(y) ||
        (final_state && !aligned16(final_state)))
        return SSD_ERR_ALIGNMENT;
    Args a = make_args(b, l, workspace);
    a.x = x;
    a.raw = raw_dt;
    a.B = B;
    a.C = C;
    a.cu = cu_seqlens;
    a.y = y;
    a.final_state = final_state;
    a.h0 = initial_state;
    // the segment-table kernel resets the header and writes the final states that no
    // segment writes
    Launch L;
    L.stream = s;
    cudaError_t e = b.tc ? tc_forward(b, a, L) : simt_forward(b, a, L);
    g_last_launches = L.count;
    return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

ssd_status_t ssd_forward(const ssd_problem_t* prob, const void* x, const float* raw_dt,
                         const void* B, const void* C, const int32_t* cu_seqlens, void* y,
                         float* final_state, void* workspace, size_t workspace_bytes,
                         void* stream) {
    return ssd_forward_state(prob, x, raw_dt, B, C, cu_seqlens, nullptr, y, final_state,
                             workspace, workspace_bytes, stream);
}

}  // extern "C"

namespace {

ssd_status_t backward_impl(const ssd_problem_t* prob, const void* x, const float* raw_dt,
                           const void* B, const void* C, const int32_t* cu_seqlens,
                           const float* h0, const void* dy, const float* dhT, void* dx,
                           float* d_raw_dt, void* dB, void* dC, float* dh0, void* workspace,
                           size_t workspace_bytes, void* stream, bool after_forward) {
    g_last_launches = 0;
    Prob b;
    Layout l;
    ssd_status_t st = check_common(prob, cu_seqlens, workspace, workspace_bytes, true, &b, &l);
    if (st != SSD_OK) return st;
    if ((h0 && !aligned16(h0)) || (dhT && !aligned16(dhT)) || (dh0 && !aligned16(dh0)))
        return SSD_ERR_ALIGNMENT;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (b.T == 0) {  // no tokens: the initial state's gradient is the final state's
        if (dh0) {
            const size_t sbytes = sizeof(float) * (size_t)b.nseq * b.H * b.P * b.N;
            const cudaError_t e = dhT ? cudaMemcpyAsync(dh0, dhT, sbytes, cudaMemcpyDeviceToDevice, s)
                                      : cudaMemsetAsync(dh0, 0, sbytes, s);
            if (e != cudaSuccess) return SSD_ERR_CUDA;
        }
        return SSD_OK;
    }
    if (!x || !raw_dt || !B || !C || !dy || !dx || !d_raw_dt || !dB || !dC)
        return SSD_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(raw_dt) || !aligned16(B) || !aligned16(C) ||
        !aligned16(dy) || !aligned16(dx) || !aligned16(d_raw_dt) || !aligned16(dB) ||
        !aligned16(dC))
        return SSD_ERR_ALIGNMENT;
    Args a = make_args(b, l, workspace);
    a.x = x;
    a.raw = raw_dt;
    a.B = B;
    a.C = C;
    a.cu = cu_seqlens;
    a.h0 = h0;
    a.dy = dy;
    a.dhT = dhT;
    a.dx = dx;
    a.draw = d_raw_dt;
    a.dB = dB;
    a.dC = dC;
    a.dh0 = dh0;
    // the tensor-core path can take the forward's segment table, tiles, factors and
    // segment states from the workspace (its header is then kept, status included)
    // (the segment-table kernel resets the header; the tensor-core path's adjoint
    // aggregate kernel zeroes the dB / dC accumulators)
    const bool reuse = after_forward && b.tc;
    const size_t nbc = sizeof(float) * (size_t)b.T * b.G * b.N;
    if (!b.tc && (cudaMemsetAsync(a.dbacc, 0, nbc, s) != cudaSuccess ||
                  cudaMemsetAsync(a.dcacc, 0, nbc, s) != cudaSuccess))
        return SSD_ERR_CUDA;
    Launch L;
    L.stream = s;
    cudaError_t e = b.tc ? tc_backward(b, a, L, reuse) : simt_backward(b, a, L);
    if (e == cudaSuccess && dh0 && b.varlen) e = launch_empty_seq_grads(b, a, L);
    g_last_launches = L.count;
    return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // namespace

extern "C" {

ssd_status_t ssd_backward(const ssd_problem_t* prob, const void* x, const float* raw_dt,
                          const void* B, const void* C, const int32_t* cu_seqlens,
                          const void* dy, void* dx, float* d_raw_dt, void* dB, void* dC,
                          void* workspace, size_t workspace_bytes, void* stream) {
    return backward_impl(prob, x, raw_dt, B, C, cu_seqlens, nullptr, dy, nullptr, dx, d_raw_dt,
                         dB, dC, nullptr, workspace, workspace_bytes, stream, false);
}

ssd_status_t ssd_backward_after_forward(const ssd_problem_t* prob, const void* x,
                                        const float* raw_dt, const void* B, const void* C,
                                        const int32_t* cu_seqlens, const void* dy, void* dx,
                                        float* d_raw_dt, void* dB, void* dC, void* workspace,
                                        size_t workspace_bytes, void* stream) {
    return backward_impl(prob, x, raw_dt, B, C, cu_seqlens, nullptr, dy, nullptr, dx, d_raw_dt,
                         dB, dC, nullptr, workspace, workspace_bytes, stream, true);
}

ssd_status_t ssd_backward_state(const ssd_problem_t* prob, const void* x, const float* raw_dt,
                                const void* B, const void* C, const int32_t* cu_seqlens,
                                const float* initial_state, const void* dy,
                                const float* d_final_state, void* dx, float* d_raw_dt, void* dB,
                                void* dC, float* d_initial_state, int after_forward,
                                void* workspace, size_t workspace_bytes, void* stream) {
    return backward_impl(prob, x, raw_dt, B, C, cu_seqlens, initial_state, dy, d_final_state, dx,
                         d_raw_dt, dB, dC, d_initial_state, workspace, workspace_bytes, stream,
                         after_forward != 0);
}

ssd_status_t ssd_decode_step(const ssd_problem_t* prob, const float* state_in, float* state_out,
                             const void* x, const float* raw_dt, const void* B, const void* C,
                             void* y, void* stream) {
    Prob b;
    ssd_status_t st = make_prob(prob, &b);
    if (st != SSD_OK) return st;
    if (prob->nseq != 0 || prob->seqlen != 1) return SSD_ERR_INVALID_ARG;
    if (!state_in || !state_out || !x || !raw_dt || !B || !C || !y) return SSD_ERR_INVALID_ARG;
    if (!aligned16(state_in) || !aligned16(state_out) || !aligned16(x) || !aligned16(raw_dt) ||
        !aligned16(B) || !aligned16(C) || !aligned16(y))
        return SSD_ERR_ALIGNMENT;
    const long long sbytes = (long long)b.nseq * b.H * b.P * b.N * 4;
    const char* si = static_cast<const char*>(static_cast<const void*>(state_in));
    const char* so = static_cast<const char*>(static_cast<void*>(state_out));
    if (si != so && si < so + sbytes && so < si + sbytes) return SSD_ERR_INVALID_ARG;
    g_last_launches = 1;
    return launch_decode_step(b, state_in, state_out, x, raw_dt, B, C, y,
                              static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? SSD_OK
               : SSD_ERR_CUDA;
}

ssd_status_t ssd_device_status(const void* workspace, void* stream, int32_t* device_status) {
    if (!workspace || !device_status) return SSD_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int v = 0;
    if (cudaMemcpyAsync(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return SSD_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SSD_ERR_CUDA;
    *device_status = v;
    return SSD_OK;
}

ssd_status_t ssd_profiler_enable(int on) {
    if (!on && g_prof_on) prof_flush();
    g_prof_on = on != 0;
    return SSD_OK;
}

ssd_status_t ssd_profiler_only(const char* name) {
    g_prof_only = name ? name : "";
    return SSD_OK;
}

void ssd_profiler_reset(void) {
    prof_flush();
    g_prof_totals.clear();
}

int ssd_profiler_count(void) {
    prof_flush();
    return (int)g_prof_totals.size();
}

ssd_status_t ssd_profiler_entry(int index, const char** name, int64_t* launches,
                                double* total_ms) {
    prof_flush();
    if (index < 0 || index >= (int)g_prof_totals.size()) return SSD_ERR_INVALID_ARG;
    const ProfTotal& t = g_prof_totals[index];
    if (name) *name = t.name.c_str();
    if (launches) *launches = t.launches;
    if (total_ms) *total_ms = t.ms;
    return SSD_OK;
}

}  // extern "C"
