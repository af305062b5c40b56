// Tensor-core (tcgen05) contraction of the TIDE router for large batches.
#include "common.cuh"

namespace tee {

size_t router_tc_scratch_bytes(int n, int d, int b) {
    (void)n; (void)d; (void)b;
    return 0;
}

tee_status router_dots_tc(int n, int d, int b, int dtype, const void* h, int64_t ldh, const void* gamma,
                          const void* w_down, float* dots, float* sumsq, void* ws, size_t ws_off, size_t ws_bytes,
                          cudaStream_t stream) {
    (void)n; (void)d; (void)b; (void)dtype; (void)h; (void)ldh; (void)gamma; (void)w_down; (void)dots;
    (void)sumsq; (void)ws; (void)ws_off; (void)ws_bytes; (void)stream;
    return TEE_ERR_UNSUPPORTED;
}

}  // namespace tee
