// ssd_step_host: one forward + backward step (or a forward alone) on host buffers.  The
// inputs are copied into a caller-owned device region, ssd_forward and
// ssd_backward_after_forward run there, and the results are copied back, all ordered on
// the caller's stream.  The copies fan out
// over library-owned copy streams (two per direction: one copy at a time per direction
// leaves part of the host link idle), joined back into the caller's stream with events.
#include <cuda_runtime.h>

#include <mutex>

#include "ssd.h"

namespace {

constexpr size_t kAlign = 256;
size_t up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// Regions of the device buffer; the workspace comes first, so that ssd_device_status can
// read the step's status from the buffer's base address.
struct StepLayout {
    size_t ws_bytes;
    size_t ws, x, raw, B, C, dy, cu, y, fs, dx, draw, dB, dC, total;
    size_t nx, nraw, nbc, ncu, nfs;
};

ssd_status_t step_layout(const ssd_problem_t* p, StepLayout* L) {
    ssd_status_t st = ssd_workspace_size(p, 1, &L->ws_bytes);
    if (st != SSD_OK) return st;
    const size_t es = p->dtype == SSD_DTYPE_BF16 ? 2 : 4;
    const size_t T = (size_t)p->batch * (size_t)p->seqlen;
    const size_t H = p->nheads, P = p->headdim, N = p->dstate, G = p->ngroups;
    L->nx = T * H * P * es;
    L->nraw = T * H * sizeof(float);
    L->nbc = T * G * N * es;
    L->ncu = p->nseq > 0 ? ((size_t)p->nseq + 1) * sizeof(int32_t) : 0;
    L->nfs = (size_t)(p->nseq > 0 ? p->nseq : p->batch) * H * P * N * sizeof(float);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = up(off + bytes);
        return at;
    };
    L->ws = take(L->ws_bytes);
    L->x = take(L->nx);
    L->raw = take(L->nraw);
    L->B = take(L->nbc);
    L->C = take(L->nbc);
    L->dy = take(L->nx);
    L->cu = take(L->ncu);
    L->y = take(L->nx);
    L->fs = take(L->nfs);
    L->dx = take(L->nx);
    L->draw = take(L->nraw);
    L->dB = take(L->nbc);
    L->dC = take(L->nbc);
    L->total = off;
    return SSD_OK;
}

// Copy streams and the events that fork and join them, per device.  One host thread at a
// time enqueues a step (an event may be recorded again as soon as the waits on its last
// record have been enqueued).
constexpr int kMaxDevices = 64;
struct CopyEngine {
    std::mutex mu;
    bool ready = false;
    cudaStream_t h2d[2], d2h[2];
    cudaEvent_t fork, in_fwd[2], in_dy, fwd_done, bwd_done, side[4];
};
CopyEngine g_engines[kMaxDevices];

bool init_engine(CopyEngine& e) {
    if (e.ready) return true;
    for (int i = 0; i < 2; ++i) {
        if (cudaStreamCreateWithFlags(&e.h2d[i], cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&e.d2h[i], cudaStreamNonBlocking) != cudaSuccess)
            return false;
    }
    cudaEvent_t* evs[] = {&e.fork,     &e.in_fwd[0], &e.in_fwd[1], &e.in_dy, &e.fwd_done,
                          &e.bwd_done, &e.side[0],   &e.side[1],   &e.side[2], &e.side[3]};
    for (cudaEvent_t* ev : evs)
        if (cudaEventCreateWithFlags(ev, cudaEventDisableTiming) != cudaSuccess) return false;
    e.ready = true;
    return true;
}

bool copy(void* dst, const void* src, size_t bytes, cudaStream_t s) {
    return bytes == 0 || cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDefault, s) == cudaSuccess;
}

}  // namespace

extern "C" {

ssd_status_t ssd_step_host_size(const ssd_problem_t* prob, size_t* bytes) {
    if (!prob || !bytes) return SSD_ERR_INVALID_ARG;
    StepLayout L;
    ssd_status_t st = step_layout(prob, &L);
    if (st != SSD_OK) return st;
    *bytes = L.total;
    return SSD_OK;
}

ssd_status_t ssd_step_host(const ssd_problem_t* prob, const void* x, const float* raw_dt,
                           const void* B, const void* C, const int32_t* cu_seqlens,
                           const void* dy, void* y, float* final_state, void* dx,
                           float* d_raw_dt, void* dB, void* dC, void* device,
                           size_t device_bytes, void* stream) {
    if (!prob) return SSD_ERR_INVALID_ARG;
    StepLayout L;
    ssd_status_t st = step_layout(prob, &L);
    if (st != SSD_OK) return st;
    if ((prob->nseq > 0) != (cu_seqlens != nullptr)) return SSD_ERR_INVALID_ARG;
    if (!device) return SSD_ERR_WORKSPACE;
    if ((uintptr_t)device % kAlign) return SSD_ERR_ALIGNMENT;
    if (device_bytes < L.total) return SSD_ERR_WORKSPACE;
    const bool bwd = dy != nullptr;  // NULL dy: forward only
    if (L.nx > 0 && (!x || !raw_dt || !B || !C || !y)) return SSD_ERR_INVALID_ARG;
    if (L.nx > 0 && bwd && (!dx || !d_raw_dt || !dB || !dC)) return SSD_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return SSD_ERR_CUDA;
    CopyEngine& e = g_engines[dev];
    std::lock_guard<std::mutex> lock(e.mu);
    if (!init_engine(e)) return SSD_ERR_CUDA;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* d = static_cast<char*>(device);
    void* ws = d + L.ws;
    void *dx_in = d + L.x, *draw_in = d + L.raw, *dB_in = d + L.B, *dC_in = d + L.C;
    void *ddy = d + L.dy, *dcu = d + L.cu, *dy_out = d + L.y, *dfs = d + L.fs;
    void *ddx = d + L.dx, *ddraw = d + L.draw, *ddB = d + L.dB, *ddC = d + L.dC;
    const int32_t* cu_dev = cu_seqlens ? static_cast<const int32_t*>(dcu) : nullptr;

    // Every internal stream rejoins the caller's stream before this returns, also on an
    // error, so that the caller's next use of the buffers is ordered after the copies.
    auto join = [&]() {
        cudaStream_t all[4] = {e.h2d[0], e.h2d[1], e.d2h[0], e.d2h[1]};
        for (int i = 0; i < 4; ++i) {
            cudaEventRecord(e.side[i], all[i]);
            cudaStreamWaitEvent(s, e.side[i], 0);
        }
    };
    bool ok = cudaEventRecord(e.fork, s) == cudaSuccess;
    for (int i = 0; i < 2 && ok; ++i)
        ok = cudaStreamWaitEvent(e.h2d[i], e.fork, 0) == cudaSuccess &&
             cudaStreamWaitEvent(e.d2h[i], e.fork, 0) == cudaSuccess;
    // inputs of the forward: x on one copy stream; raw_dt, B, C, cu_seqlens on the other,
    // then dy there (the backward waits for it; it moves while the forward runs)
    ok = ok && copy(dx_in, x, L.nx, e.h2d[0]) &&
         cudaEventRecord(e.in_fwd[0], e.h2d[0]) == cudaSuccess;
    ok = ok && copy(draw_in, raw_dt, L.nraw, e.h2d[1]) && copy(dB_in, B, L.nbc, e.h2d[1]) &&
         copy(dC_in, C, L.nbc, e.h2d[1]) && copy(dcu, cu_seqlens, L.ncu, e.h2d[1]) &&
         cudaEventRecord(e.in_fwd[1], e.h2d[1]) == cudaSuccess;
    if (bwd)
        ok = ok && copy(ddy, dy, L.nx, e.h2d[1]) &&
             cudaEventRecord(e.in_dy, e.h2d[1]) == cudaSuccess;
    ok = ok && cudaStreamWaitEvent(s, e.in_fwd[0], 0) == cudaSuccess &&
         cudaStreamWaitEvent(s, e.in_fwd[1], 0) == cudaSuccess;
    if (!ok) {
        join();
        return SSD_ERR_CUDA;
    }
    st = ssd_forward(prob, dx_in, static_cast<const float*>(draw_in), dB_in, dC_in, cu_dev,
                     dy_out, final_state ? static_cast<float*>(dfs) : nullptr, ws, L.ws_bytes,
                     stream);
    if (st != SSD_OK) {
        join();
        return st;
    }
    // y and final_state go out while the backward runs
    ok = cudaEventRecord(e.fwd_done, s) == cudaSuccess &&
         cudaStreamWaitEvent(e.d2h[0], e.fwd_done, 0) == cudaSuccess &&
         copy(y, dy_out, L.nx, e.d2h[0]) &&
         (!final_state || copy(final_state, dfs, L.nfs, e.d2h[0]));
    if (!ok || !bwd) {
        join();
        return ok ? SSD_OK : SSD_ERR_CUDA;
    }
    if (cudaStreamWaitEvent(s, e.in_dy, 0) != cudaSuccess) {
        join();
        return SSD_ERR_CUDA;
    }
    st = ssd_backward_after_forward(prob, dx_in, static_cast<const float*>(draw_in), dB_in, dC_in,
                                    cu_dev, ddy, ddx, static_cast<float*>(ddraw), ddB, ddC, ws,
                                    L.ws_bytes, stream);
    if (st != SSD_OK) {
        join();
        return st;
    }
    ok = cudaEventRecord(e.bwd_done, s) == cudaSuccess;
    for (int i = 0; i < 2 && ok; ++i)
        ok = cudaStreamWaitEvent(e.d2h[i], e.bwd_done, 0) == cudaSuccess;
    ok = ok && copy(dx, ddx, L.nx, e.d2h[1]) && copy(d_raw_dt, ddraw, L.nraw, e.d2h[0]) &&
         copy(dB, ddB, L.nbc, e.d2h[0]) && copy(dC, ddC, L.nbc, e.d2h[0]);
    join();
    return ok ? SSD_OK : SSD_ERR_CUDA;
}

}  // extern "C"
