// Library-wide entry points: version, status strings, workspace set-up and
// the device fault word.
#include <atomic>

#include "common.cuh"
#include "tc.cuh"

namespace tee {

static thread_local int g_last_cuda = 0;
static std::atomic<uint64_t> g_launches{0};

tee_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return TEE_OK;
    g_last_cuda = static_cast<int>(e);
    return TEE_ERR_CUDA;
}

tee_status launch_status() {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return cuda_status(cudaGetLastError());
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
    return n;
}

namespace {
// The failure-detection path of the pipelines' waits: one block waits on an
// mbarrier that nothing completes. Every wait gives up after limit_ns, the first
// records TEE_DEVERR_TIMEOUT (detail 99) in the workspace header, and the kernel
// returns; the context stays usable.
constexpr int CHECK_WHERE = 99;
__global__ void __launch_bounds__(64) wait_timeout_check_kernel(uint64_t limit_ns, void* ws) {
    __shared__ uint64_t bar;
    __shared__ volatile int abort;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);
        abort = 0;
        tc::fence_barrier_init();
    }
    __syncthreads();
    (void)tc::mbar_wait_for(&bar, 0, &abort, ws, CHECK_WHERE, limit_ns, 1000);
}
}  // namespace

}  // namespace tee

using namespace tee;

extern "C" {

const char* tee_version(void) { return "tee 0.1 (sm_103a)"; }

const char* tee_status_string(tee_status s) {
    switch (s) {
        case TEE_OK: return "ok";
        case TEE_ERR_INVALID_ARG: return "invalid argument";
        case TEE_ERR_UNSUPPORTED: return "unsupported dtype or format";
        case TEE_ERR_CUDA: return "CUDA error";
        case TEE_ERR_WORKSPACE: return "workspace too small";
        case TEE_ERR_DEVICE: return "device fault recorded";
    }
    return "unknown status";
}

int tee_last_cuda_error(void) { return g_last_cuda; }

uint64_t tee_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

tee_status tee_workspace_init(void* ws, size_t bytes, void* stream) {
    if (!ws || bytes < TEE_WS_HEADER_BYTES) return TEE_ERR_WORKSPACE;
    return cuda_status(cudaMemsetAsync(ws, 0, bytes, static_cast<cudaStream_t>(stream)));
}

tee_status tee_get_device_error(const void* ws, int32_t* code, int32_t* detail, void* stream) {
    if (!ws) return TEE_ERR_WORKSPACE;
    int32_t h[2] = {0, 0};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    tee_status st = cuda_status(cudaMemcpyAsync(h, ws, sizeof(h), cudaMemcpyDeviceToHost, s));
    if (st != TEE_OK) return st;
    st = cuda_status(cudaStreamSynchronize(s));
    if (st != TEE_OK) return st;
    if (code) *code = h[0];
    if (detail) *detail = h[1];
    return h[0] ? TEE_ERR_DEVICE : TEE_OK;
}

tee_status tee_check_wait_timeout(void* ws, uint32_t limit_us, void* stream) {
    if (!ws) return TEE_ERR_WORKSPACE;
    if (limit_us == 0 || limit_us > 100000) return TEE_ERR_INVALID_ARG;
    wait_timeout_check_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(uint64_t(limit_us) * 1000, ws);
    return launch_status();
}

tee_status tee_clear_device_error(void* ws, void* stream) {
    if (!ws) return TEE_ERR_WORKSPACE;
    return cuda_status(cudaMemsetAsync(ws, 0, TEE_WS_HEADER_BYTES, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
