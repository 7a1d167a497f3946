// ssd_forward_noalloc: the forward scan for callers that cannot allocate
// device memory.  Its scratch lives in one file-scope device array; the
// entry point finds that array's device address once per device and hands it
// to the unchanged ssd_forward as the workspace.
#include <mutex>

#include "ssd_internal.cuh"

// The scratch itself.  In host code this name is only a host-side stand-in,
// never a device address: the address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SSD_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up on the
// first call for that device).
ssd_status_t noalloc_scratch(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return SSD_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return SSD_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p)
            return SSD_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return SSD_OK;
}

}  // namespace

extern "C" ssd_status_t ssd_forward_noalloc(const ssd_problem_t* prob, const void* x,
                                            const float* raw_dt, const void* B, const void* C,
                                            const int32_t* cu_seqlens, void* y,
                                            float* final_state, void* stream) {
    size_t need = 0;
    ssd_status_t st = ssd_workspace_size(prob, 0, &need);
    if (st != SSD_OK) return st;
    if (need > (size_t)SSD_NOALLOC_SCRATCH_BYTES) return SSD_ERR_WORKSPACE;
    void* scratch = nullptr;
    st = noalloc_scratch(&scratch);
    if (st != SSD_OK) return st;
    return ssd_forward(prob, x, raw_dt, B, C, cu_seqlens, y, final_state, scratch,
                       (size_t)SSD_NOALLOC_SCRATCH_BYTES, stream);
}

// The status word sits at the start of the scratch array, where every workspace keeps it.
extern "C" ssd_status_t ssd_forward_noalloc_status(void* stream, int32_t* device_status) {
    if (!device_status) return SSD_ERR_INVALID_ARG;
    void* scratch = nullptr;
    ssd_status_t st = noalloc_scratch(&scratch);
    if (st != SSD_OK) return st;
    return ssd_device_status(scratch, stream, device_status);
}
