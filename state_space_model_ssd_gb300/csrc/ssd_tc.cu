// Tensor-core path (bf16, P = 64, N in {64, 128}, chunk 64).
#include "ssd_device.cuh"

namespace ssd {

bool tc_supported(int dtype, int P, int N, int Q) {
    (void)dtype; (void)P; (void)N; (void)Q;
    return false;
}

cudaError_t tc_forward(const Prob&, const Args&, Launch&) { return cudaErrorNotSupported; }
cudaError_t tc_backward(const Prob&, const Args&, Launch&) { return cudaErrorNotSupported; }

}  // namespace ssd
