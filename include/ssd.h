/*
 * ssd.h -- C ABI of the SSD selective-state scan library (libssd.so, sm_103a).
 *
 * The operation (page "Mamba-2架构与LaCT并行计算技术解析", §1.1, the state
 * equations, and §1.2, independent heads): for every head h and every token t
 *
 *     delta_t = softplus(raw_dt_t + delta_init)
 *     H_t     = exp(-delta_t) * H_{t-1} + delta_t * x_t B_t^T       (H is P x N, fp32)
 *     y_t     = H_t C_t
 *
 * with H = 0 before the first token of every sequence (the zero-initial-state
 * note under the same equations).  The library evaluates it in the chunked,
 * semiseparable way of page "长序列 Mamba 多卡训练算力和显存怎么同时省" §一:
 * diagonal blocks inside each chunk, a small state passed between chunks.
 * Packed variable-length input follows the cu_seqlens convention of the same
 * page, §三: the state restarts at every sequence boundary.
 *
 * General rules for every entry point:
 *  - All tensor arguments are DEVICE pointers on the current CUDA device,
 *    contiguous, row-major, 16-byte aligned (ssd_step_host alone takes host
 *    buffers).  The caller owns every buffer; the library allocates nothing on
 *    the device and keeps no pointer after a call returns.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream).  No call synchronises except ssd_device_status().
 *  - Host-side argument checks run before any launch; on failure nothing is
 *    launched and a nonzero ssd_status_t is returned.  Errors that only the
 *    device can see (a malformed cu_seqlens array) are recorded in a status
 *    word inside the workspace and read with ssd_device_status().
 *  - Calls that share a workspace must not overlap on the GPU.
 *
 * Layouts (T = batch * seqlen tokens, H heads, P = headdim, N = dstate,
 * G = ngroups; head h reads B/C group h / (H / G)):
 *     x, y, dy, dx     [T][H][P]   dtype = problem.dtype
 *     raw_dt, d_raw_dt [T][H]      float32
 *     B, C, dB, dC     [T][G][N]   dtype = problem.dtype
 *     final_state      [nseq or batch][H][P][N] float32
 *     cu_seqlens       [nseq + 1]  int32, cu[0] = 0, cu[nseq] = T, non-decreasing
 */
#ifndef SSD_H_
#define SSD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SSD_API_VERSION 1

typedef enum {
    SSD_OK = 0,
    SSD_ERR_INVALID_ARG = 1,   /* null pointer, bad size or inconsistent problem */
    SSD_ERR_UNSUPPORTED = 2,   /* valid problem outside the supported shape set */
    SSD_ERR_ALIGNMENT = 3,     /* a pointer is not 16-byte aligned (workspace: 256) */
    SSD_ERR_WORKSPACE = 4,     /* workspace missing or smaller than ssd_workspace_size(); as a
                                  device status: the workspace does not hold the forward that
                                  ssd_backward_after_forward was told to reuse */
    SSD_ERR_CUDA = 5,          /* a CUDA runtime call failed (launch error) */
    SSD_ERR_TIMEOUT = 6,       /* a bounded device-side wait gave up (device status) */
    SSD_ERR_DEVICE = 7         /* device-side check failed, e.g. bad cu_seqlens (device status) */
} ssd_status_t;

typedef enum { SSD_DTYPE_F32 = 0, SSD_DTYPE_BF16 = 1 } ssd_dtype_t;

typedef struct {
    int64_t batch;       /* rows of a dense batch; must be 1 when cu_seqlens is used */
    int64_t seqlen;      /* tokens per row; with cu_seqlens: total packed tokens T */
    int32_t nheads;      /* H */
    int32_t headdim;     /* P */
    int32_t dstate;      /* N */
    int32_t ngroups;     /* G, divides H (B and C are shared by H / G heads) */
    int32_t chunk_size;  /* Q, the diagonal-block length; the result does not depend on it */
    int32_t nseq;        /* 0: dense batch; > 0: number of packed sequences in cu_seqlens */
    float delta_init;    /* added to raw_dt before softplus (e.g. -4.6) */
    int32_t dtype;       /* ssd_dtype_t of x, B, C, y, dy, dx, dB, dC */
} ssd_problem_t;

/* Supported shapes: P in {8,16,32,64,128}; N in {8,16,32,64,128};
 * chunk_size in {16,32,64,128,256}; T <= 2^31 - 1; G divides H.
 * bf16 problems with P = 64, N in {64,128}, chunk_size = 64 and at least chunk_size
 * tokens in all run on the tensor-core path (any number of heads per group); every
 * other supported problem runs on the SIMT path. */

/* Bytes of device workspace that ssd_forward (for_backward = 0) or
 * ssd_backward (for_backward = 1) needs for `prob`.  Host function, no launch; on the
 * tensor-core path with dense rows the segment length, and with it the size, follows
 * the current device's SM count, so query it with the device current that will run
 * the calls.  Returns SSD_ERR_INVALID_ARG / SSD_ERR_UNSUPPORTED for a bad problem. */
ssd_status_t ssd_workspace_size(const ssd_problem_t* prob, int for_backward, size_t* bytes);

/* Forward scan.  Reads x, raw_dt, B, C (and cu_seqlens when prob->nseq > 0,
 * else it must be NULL); writes y and, when final_state is not NULL, the
 * state after the last token of every sequence (row) -- the quantity that
 * crosses from one chunk to the next, page "长序列 Mamba 多卡训练算力和显存
 * 怎么同时省" §一.  workspace: >= ssd_workspace_size(prob, 0) bytes, 256-byte
 * aligned, contents ignored on entry. */
ssd_status_t ssd_forward(const ssd_problem_t* prob, const void* x, const float* raw_dt,
                         const void* B, const void* C, const int32_t* cu_seqlens, void* y,
                         float* final_state, void* workspace, size_t workspace_bytes,
                         void* stream);

/* ssd_forward from a given state per sequence: H = initial_state[seq] before the first
 * token of every sequence (dense row) instead of zero -- the carried-over state of page
 * "Mamba-2架构与LaCT并行计算技术解析" §1.1 (the note on initialising H from the previous
 * frame's final state).  initial_state: [nseq or batch][H][P][N] float32 device memory,
 * 16-byte aligned, or NULL for zero (then this is ssd_forward).  The final state of an
 * empty packed sequence is its initial state. */
ssd_status_t ssd_forward_state(const ssd_problem_t* prob, const void* x, const float* raw_dt,
                               const void* B, const void* C, const int32_t* cu_seqlens,
                               const float* initial_state, void* y, float* final_state,
                               void* workspace, size_t workspace_bytes, void* stream);

/* Backward of ssd_forward for an upstream gradient dy of y (the gradient of
 * final_state is taken as zero).  Writes dx [T][H][P], d_raw_dt [T][H]
 * (float32, includes the softplus derivative), dB and dC [T][G][N] (summed
 * over the heads of each group, fp32 accumulation, one rounding to dtype).
 * Reverse-mode derivative of the recurrence of page "Mamba-2架构与LaCT并行
 * 计算技术解析" §1.1; the forward states are recomputed, per the
 * recompute-from-checkpoints idea of that page's §4.1.  workspace: >=
 * ssd_workspace_size(prob, 1) bytes, 256-byte aligned. */
ssd_status_t ssd_backward(const ssd_problem_t* prob, const void* x, const float* raw_dt,
                          const void* B, const void* C, const int32_t* cu_seqlens,
                          const void* dy, void* dx, float* d_raw_dt, void* dB, void* dC,
                          void* workspace, size_t workspace_bytes, void* stream);

/* ssd_backward for the workspace that the preceding ssd_forward call used, on the same
 * stream, with the same problem and the same x, raw_dt, B, C (and cu_seqlens) buffers,
 * whose contents have not changed since.  On the tensor-core path it takes the
 * forward's segment table, masked C B^T tiles, chunk factors and segment states from the
 * workspace instead of recomputing them (activations saved by the forward, in the
 * sense of page "Mamba-2架构与LaCT并行计算技术解析" §4.1); the results are those of
 * ssd_backward.  The forward records its problem and input pointers (initial_state
 * included) in the workspace;
 * if they differ from this call's, the device status becomes SSD_ERR_WORKSPACE and no
 * gradient is computed (ssd_device_status reports it).  Buffer contents are not
 * compared: changing them between the two calls gives the gradient at the old inputs.
 * The forward's own device status is kept.  On the SIMT path this call is ssd_backward.
 * workspace: >= ssd_workspace_size(prob, 1) bytes, passed to the forward as well. */
ssd_status_t ssd_backward_after_forward(const ssd_problem_t* prob, const void* x,
                                        const float* raw_dt, const void* B, const void* C,
                                        const int32_t* cu_seqlens, const void* dy, void* dx,
                                        float* d_raw_dt, void* dB, void* dC, void* workspace,
                                        size_t workspace_bytes, void* stream);

/* Backward of ssd_forward_state: the gradient of
 *     L = sum_t dy_t . y_t + sum_seq <d_final_state[seq], final_state[seq]>
 * with respect to x, raw_dt, B, C (written as by ssd_backward) and, when d_initial_state is
 * not NULL, to initial_state: d_initial_state[seq] = dL / dH before the sequence's first
 * token ([nseq or batch][H][P][N] float32; an empty sequence's is its d_final_state).
 * initial_state (NULL: zero) must be the one the forward used; d_final_state ([nseq or
 * batch][H][P][N] float32, NULL: zero) is the upstream gradient of final_state.  Reverse
 * mode of the recurrence of page "Mamba-2架构与LaCT并行计算技术解析" §1.1.
 * after_forward != 0: as ssd_backward_after_forward (the preceding ssd_forward_state on the
 * same workspace, inputs and initial_state); 0: as ssd_backward.  workspace: >=
 * ssd_workspace_size(prob, 1) bytes. */
ssd_status_t ssd_backward_state(const ssd_problem_t* prob, const void* x, const float* raw_dt,
                                const void* B, const void* C, const int32_t* cu_seqlens,
                                const float* initial_state, const void* dy,
                                const float* d_final_state, void* dx, float* d_raw_dt, void* dB,
                                void* dC, float* d_initial_state, int after_forward,
                                void* workspace, size_t workspace_bytes, void* stream);

/* Bidirectional mode (page "Mamba-2架构与LaCT并行计算技术解析" §3.1): the scan over each
 * sequence (dense row or packed sequence) and the scan over the same sequence reversed,
 * on the same x, raw_dt, B, C; the reverse direction's output is put back at its tokens'
 * positions and the two are concatenated along the last dimension:
 *     y[t][h] = [ y_forward[t][h] (P values) | y_reverse[t][h] (P values) ],
 * y_reverse[t] depending on tokens t .. the sequence's end.  y: [T][H][2P] (dtype of x).
 * final_state_fwd / final_state_rev ([nseq or batch][H][P][N] float32, NULL: not written):
 * each direction's state after its last token (the state size doubles).  workspace: >=
 * ssd_bidirectional_workspace_size(prob, 0) bytes, 256-byte aligned; it holds the
 * reversed inputs and both directions' outputs besides ssd_forward's workspace. */
ssd_status_t ssd_bidirectional_workspace_size(const ssd_problem_t* prob, int for_backward,
                                              size_t* bytes);
ssd_status_t ssd_bidirectional_forward(const ssd_problem_t* prob, const void* x,
                                       const float* raw_dt, const void* B, const void* C,
                                       const int32_t* cu_seqlens, void* y,
                                       float* final_state_fwd, float* final_state_rev,
                                       void* workspace, size_t workspace_bytes, void* stream);
/* Backward of ssd_bidirectional_forward for an upstream gradient dy [T][H][2P] of y (zero
 * final-state gradients): dx, d_raw_dt, dB, dC as ssd_backward writes them, each the sum of
 * the two directions' contributions.  workspace: >= ssd_bidirectional_workspace_size(prob,
 * 1) bytes. */
ssd_status_t ssd_bidirectional_backward(const ssd_problem_t* prob, const void* x,
                                        const float* raw_dt, const void* B, const void* C,
                                        const int32_t* cu_seqlens, const void* dy, void* dx,
                                        float* d_raw_dt, void* dB, void* dC, void* workspace,
                                        size_t workspace_bytes, void* stream);

/* One token of the recurrence for every sequence of a batch (single-token decode), from
 * a carried state (page "Mamba-2架构与LaCT并行计算技术解析" §1.1):
 *     delta = softplus(raw_dt + delta_init),
 *     state <- exp(-delta) state + delta x B^T,   y = state C.
 * prob: batch = number of sequences, seqlen = 1, nseq = 0; H, P, N, G, dtype, delta_init
 * as for ssd_forward (chunk_size must be a supported value and is otherwise unused).
 * state_in, state_out: [batch][H][P][N] float32 (the same pointer updates in place; other
 * overlaps are SSD_ERR_INVALID_ARG); x, y: [batch][H][P]; raw_dt: [batch][H] float32;
 * B, C: [batch][G][N].  Device memory, 16-byte aligned; no workspace.  Bound by the
 * state's bytes: it is read and written once. */
ssd_status_t ssd_decode_step(const ssd_problem_t* prob, const float* state_in, float* state_out,
                             const void* x, const float* raw_dt, const void* B, const void* C,
                             void* y, void* stream);

/* Device bytes that ssd_step_host needs for `prob`: the backward workspace followed by
 * device copies of the step's inputs and results.  Pure host function. */
ssd_status_t ssd_step_host_size(const ssd_problem_t* prob, size_t* bytes);

/* One forward + backward step on HOST buffers (the layouts above, in host memory):
 * x, raw_dt, B, C, cu_seqlens (a host array; NULL for a dense batch) and dy are read from
 * host memory; y, final_state (NULL: not written), dx, d_raw_dt, dB and dC are written to
 * host memory.  With dy = NULL the step is the forward alone (dx, d_raw_dt, dB and dC
 * are then not used and may be NULL).  The call copies the inputs into `device` (>= ssd_step_host_size bytes of
 * device memory owned by the caller, 256-byte aligned), runs ssd_forward and
 * ssd_backward_after_forward there, and copies the results back.  Asynchronous on
 * `stream` like every other call: the host outputs are complete once the stream has
 * passed the call (e.g. after cudaStreamSynchronize), and every host buffer must stay
 * valid until then.  Page-locked host memory lets the copies run asynchronously
 * (pageable memory is staged synchronously by the CUDA runtime).  Inside a call, dy is
 * copied in while the forward runs and y and final_state out while the backward runs,
 * on copy streams the library creates once per device; each call is ordered after the
 * caller's earlier work on `stream` and the caller's later work after all of it.  Two
 * calls on different streams with different `device` buffers overlap one step's copies
 * with the other's kernels.  The workspace is the first region of `device`, so
 * ssd_device_status(device, ...) reads the step's device status.  Errors: those of
 * ssd_forward and ssd_backward; SSD_ERR_WORKSPACE if `device` is NULL or smaller than
 * ssd_step_host_size(); SSD_ERR_ALIGNMENT if it is not 256-byte aligned; SSD_ERR_CUDA if
 * a copy or an event could not be enqueued.  One host thread at a time enqueues a step
 * (calls from several threads are serialised). */
ssd_status_t ssd_step_host(const ssd_problem_t* prob, const void* x, const float* raw_dt,
                           const void* B, const void* C, const int32_t* cu_seqlens,
                           const void* dy, void* y, float* final_state, void* dx,
                           float* d_raw_dt, void* dB, void* dC, void* device,
                           size_t device_bytes, void* stream);

/* Size of the device scratch array that ssd_forward_noalloc works in. */
#define SSD_NOALLOC_SCRATCH_BYTES (64u << 20)

/* ssd_forward for callers that cannot allocate device memory.  The pages have
 * no counterpart to this call: it exists for host applications whose device
 * memory is owned by someone else -- a plugin or callback inside a framework
 * that hands out no workspace, or code on a latency-critical path where
 * cudaMalloc / cudaFree (which may synchronise the device) are not allowed.
 * Such a caller passes only inputs and outputs; the scratch that ssd_forward
 * takes as `workspace` comes instead from one SSD_NOALLOC_SCRATCH_BYTES array
 * that the library declares in device memory.  Every GPU on which the library
 * is loaded holds that array until the process exits (with CUDA's default lazy
 * module loading, from the first call on that GPU).
 *  - Same arguments, layouts and results as ssd_forward, minus the workspace.
 *  - Problems whose forward workspace (ssd_workspace_size(prob, 0)) exceeds
 *    SSD_NOALLOC_SCRATCH_BYTES are rejected with SSD_ERR_WORKSPACE before any
 *    launch.
 *  - The first call on a device looks up the array's device address for that
 *    device (the current one); make that first call before any stream capture.
 *  - Every call on a device uses the same array, which keeps the previous
 *    call's contents (the call clears what it needs cleared); calls that may
 *    overlap on the GPU, from any stream or thread, race and must be ordered
 *    by the caller.
 *  - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *  - Errors that only the device sees (a malformed cu_seqlens, a wait that timed out)
 *    go to the status word inside the array; ssd_forward_noalloc_status() reads it.
 *  - The array's address is kept per device for the life of the process: calling
 *    cudaDeviceReset() after the first call on a device is not supported. */
ssd_status_t ssd_forward_noalloc(const ssd_problem_t* prob, const void* x, const float* raw_dt,
                                 const void* B, const void* C, const int32_t* cu_seqlens,
                                 void* y, float* final_state, void* stream);

/* The device status word that the last ssd_forward_noalloc call on the current device
 * left (SSD_OK, SSD_ERR_DEVICE, SSD_ERR_TIMEOUT), read like ssd_device_status():
 * synchronises `stream` first.  Returns SSD_ERR_CUDA if that failed. */
ssd_status_t ssd_forward_noalloc_status(void* stream, int32_t* device_status);

/* Synchronises `stream` and returns in *device_status the status word that
 * the last call using `workspace` left (SSD_OK, SSD_ERR_DEVICE, SSD_ERR_TIMEOUT).
 * Returns SSD_ERR_CUDA if the synchronisation itself failed. */
ssd_status_t ssd_device_status(const void* workspace, void* stream, int32_t* device_status);

/* Which kernel path a problem takes: "tensor-core", "simt", or NULL for an
 * unsupported problem.  Pure host function. */
const char* ssd_dispatch_path(const ssd_problem_t* prob, int for_backward);

/* Number of kernels the last ssd_forward / ssd_backward call on this host
 * thread launched (memsets not counted). */
int ssd_last_launch_count(void);

/* Per-kernel timing.  While enabled, every kernel launch is bracketed by CUDA
 * events recorded on the launch stream; ssd_profiler_entry() synchronises
 * them and reports, per kernel name, the launch count and total device time.
 * Not thread-safe; meant for benchmarks. */
ssd_status_t ssd_profiler_enable(int on);
/* Restricts the timing to launches of the kernel called `name` (as reported by
 * ssd_profiler_entry); NULL times every kernel again.  Each pair of events holds the
 * launch that follows it back until the kernel before it has finished, so timing
 * only the kernel of interest leaves the other kernel boundaries of a pass alone. */
ssd_status_t ssd_profiler_only(const char* name);
void ssd_profiler_reset(void);
int ssd_profiler_count(void);
ssd_status_t ssd_profiler_entry(int index, const char** name, int64_t* launches,
                                double* total_ms);

const char* ssd_status_string(ssd_status_t status);
int ssd_version(void);

#ifdef __cplusplus
}
#endif
#endif /* SSD_H_ */
