// Tensor-core (tcgen05) path of the KV fill.
#include "fill.cuh"

namespace tee {

size_t fill_tc_prep_bytes(const tee_fill_desc& D, int n_layers) {
    (void)D;
    (void)n_layers;
    return 0;
}

tee_status fill_tc_prepare(const tee_fill_desc& D, int n_layers, const tee_fill_layer* layers, char* tc_area,
                           cudaStream_t s) {
    (void)D; (void)n_layers; (void)layers; (void)tc_area; (void)s;
    return TEE_OK;
}

size_t fill_tc_ws_bytes(const tee_fill_desc& D, int n_layers, int n_max) {
    (void)D; (void)n_layers; (void)n_max;
    return 0;
}

tee_status fill_tc_run(const FillCall& fc) {
    (void)fc;
    return TEE_ERR_UNSUPPORTED;
}

}  // namespace tee
