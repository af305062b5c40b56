// A whole decode step from host buffers to host buffers in one call: the
// inputs' host-to-device copies, the front (gate + compaction + exit scatter)
// and the KV fill of the exiting tokens, and the results' copies back. It only
// sequences the library's own calls. The sequence is captured once into a CUDA
// graph on the step's own stream and replayed while the token count and the
// host buffers stay the same (a serving loop's case), so that a step costs the
// host one graph launch; the caller's stream and the step's stream are ordered
// by two events. Where capture is refused (pageable host memory, for one) the
// sequence is enqueued directly on the caller's stream instead.
// When every host buffer is page-locked memory that the device reaches directly
// (mapped into its address space, as page-locked memory is under unified
// addressing), one copy kernel reads all the inputs and another writes all the
// results: two launches instead of eight copies, whose fixed costs would add up
// on the step's critical path. Otherwise the copies are cudaMemcpyAsync calls.
#include <new>

#include "common.cuh"

struct tee_decode_step {
    tee_gate_desc gate;
    int n_max;
    tee_fill_desc fill;
    int n_layers;
    tee_fill_layer* layers;   // owned copy
    const void* prep;
    size_t prep_bytes;
    void* k_cache;
    void* v_cache;
    tee_cache_layout cache;
    tee_step_buffers buf;
    // the captured sequence and the arguments it was captured for
    cudaStream_t cap;
    cudaEvent_t ev_in, ev_out;
    cudaGraphExec_t exec;
    bool graph_refused;
    int g_n;
    const void* g_ptr[8];
};

using namespace tee;

extern "C" tee_status tee_decode_step_create(const tee_gate_desc* gate, int32_t n_max, const tee_fill_desc* fill,
                                             int32_t n_layers, const tee_fill_layer* layers, const void* fill_prep,
                                             size_t fill_prep_bytes, void* k_cache, void* v_cache,
                                             const tee_cache_layout* cache, const tee_step_buffers* buf,
                                             tee_decode_step** step) {
    if (!gate || !fill || !cache || !buf || !step || n_max <= 0 || n_layers < 0 || (n_layers > 0 && !layers))
        return TEE_ERR_INVALID_ARG;
    if (gate->mode != TEE_GATE_COSINE || gate->d != fill->d || gate->dtype != fill->dtype) return TEE_ERR_INVALID_ARG;
    if (!buf->h_prev || !buf->h_cur || !buf->pos || !buf->score || !buf->mask || !buf->cont_rows || !buf->exit_rows ||
        !buf->out || !buf->counts || buf->n_out < 0 || !fill_prep || !k_cache || !v_cache)
        return TEE_ERR_INVALID_ARG;
    const size_t need_front = tee_exit_gate_compact_scatter_workspace_size(gate, n_max);
    const size_t need_fill = tee_kv_fill_workspace_size(fill, n_layers, n_max);
    if (need_front == 0 || need_fill == 0) return TEE_ERR_INVALID_ARG;
    if (!buf->ws || buf->ws_bytes < need_front || buf->ws_bytes < need_fill) return TEE_ERR_WORKSPACE;
    tee_decode_step* s = new (std::nothrow) tee_decode_step;
    if (!s) return TEE_ERR_INVALID_ARG;
    s->layers = n_layers > 0 ? new (std::nothrow) tee_fill_layer[n_layers] : nullptr;
    if (n_layers > 0 && !s->layers) {
        delete s;
        return TEE_ERR_INVALID_ARG;
    }
    for (int l = 0; l < n_layers; ++l) s->layers[l] = layers[l];
    s->gate = *gate;
    s->n_max = n_max;
    s->fill = *fill;
    s->n_layers = n_layers;
    s->prep = fill_prep;
    s->prep_bytes = fill_prep_bytes;
    s->k_cache = k_cache;
    s->v_cache = v_cache;
    s->cache = *cache;
    s->buf = *buf;
    s->cap = nullptr;
    s->ev_in = s->ev_out = nullptr;
    s->exec = nullptr;
    s->graph_refused = false;
    s->g_n = -1;
    if (cudaStreamCreateWithFlags(&s->cap, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&s->ev_in, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&s->ev_out, cudaEventDisableTiming) != cudaSuccess) {
        const tee_status st = cuda_status(cudaGetLastError());
        tee_decode_step_destroy(s);
        return st == TEE_OK ? TEE_ERR_CUDA : st;
    }
    *step = s;
    return TEE_OK;
}

namespace {

struct CopySeg {
    const uint8_t* src;
    uint8_t* dst;
    int64_t bytes;
};
struct CopyList {
    CopySeg seg[4];
    int n;
};

// Up to four copies in one launch, 16 bytes a thread and step where both ends
// are 16-byte aligned. Loads are volatile-cached (ld.global.cv): a replay reads
// what the host wrote since, not a line that an earlier step left in a cache.
// The next kernel may start launching at once; launched as a dependent itself
// (the results' copy after the fill), it waits for the kernel before it first.
__global__ void __launch_bounds__(256) step_copy_kernel(CopyList l) {
    allow_dependents();
    wait_prior_grid();
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t nth = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int s = 0; s < l.n; ++s) {
        const CopySeg c = l.seg[s];
        const bool v16 = ((reinterpret_cast<uintptr_t>(c.src) | reinterpret_cast<uintptr_t>(c.dst)) & 15) == 0;
        const int64_t n16 = v16 ? c.bytes / 16 : 0;
        for (int64_t i = tid; i < n16; i += nth)
            reinterpret_cast<uint4*>(c.dst)[i] = __ldcv(reinterpret_cast<const uint4*>(c.src) + i);
        for (int64_t i = n16 * 16 + tid; i < c.bytes; i += nth) c.dst[i] = __ldcv(c.src + i);
    }
}

// The device's address of page-locked host memory it reaches directly, or null.
const void* device_view(const void* p) {
    if (!p) return nullptr;
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

tee_status launch_copies(const CopyList& l, bool dependent, cudaStream_t s) {
    int64_t most = 0;
    for (int i = 0; i < l.n; ++i) most = l.seg[i].bytes > most ? l.seg[i].bytes : most;
    if (most == 0) return TEE_OK;
    const int64_t want = (most / 16 + 255) / 256;
    const int blocks = static_cast<int>(want < 1 ? 1 : (want > 4 * sm_count() ? 4 * sm_count() : want));
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = dependent ? 1 : 0;
    const tee_status st = cuda_status(cudaLaunchKernelEx(&cfg, step_copy_kernel, l));
    return st != TEE_OK ? st : launch_status();
}

// The device's views of the eight host buffers (h_prev, h_cur, pos, seq, score,
// mask, counts, out); looked up outside any stream capture.
struct HostViews {
    const void* v[8];
};
HostViews host_views(const void* const (&ptr)[8]) {
    HostViews h{};
    for (int i = 0; i < 8; ++i) h.v[i] = device_view(ptr[i]);
    return h;
}

// The step's copies and calls, enqueued on stream s.
tee_status enqueue_step(tee_decode_step* step, int n, const void* h_prev, const void* h_cur, const int32_t* pos,
                        const int32_t* seq, float* score, uint8_t* mask, int32_t* counts, void* out,
                        const HostViews& views, cudaStream_t s) {

    void* stream = s;
    const tee_step_buffers& b = step->buf;
    const int d = step->gate.d;
    const size_t row = static_cast<size_t>(d) * dtype_bytes(step->gate.dtype);
    const bool use_seq = seq && b.seq;
    // the device's view of every host buffer, or the copies go through cudaMemcpyAsync
    const void* const* hv = views.v;
    const bool mapped = hv[0] && hv[1] && hv[2] && (!use_seq || hv[3]) && (!score || hv[4]) && (!mask || hv[5]) &&
                        (!counts || hv[6]) && (!out || hv[7]);
    tee_status st = TEE_OK;
    // inputs
    if (mapped) {
        CopyList l{};
        l.seg[l.n++] = CopySeg{static_cast<const uint8_t*>(hv[0]), static_cast<uint8_t*>(b.h_prev),
                               static_cast<int64_t>(n * row)};
        l.seg[l.n++] = CopySeg{static_cast<const uint8_t*>(hv[1]), static_cast<uint8_t*>(b.h_cur),
                               static_cast<int64_t>(n * row)};
        l.seg[l.n++] = CopySeg{static_cast<const uint8_t*>(hv[2]), reinterpret_cast<uint8_t*>(b.pos),
                               static_cast<int64_t>(n * sizeof(int32_t))};
        if (use_seq)
            l.seg[l.n++] = CopySeg{static_cast<const uint8_t*>(hv[3]), reinterpret_cast<uint8_t*>(b.seq),
                                   static_cast<int64_t>(n * sizeof(int32_t))};
        st = launch_copies(l, false, s);
    } else {
        st = cuda_status(cudaMemcpyAsync(b.h_prev, h_prev, n * row, cudaMemcpyHostToDevice, s));
        if (st == TEE_OK) st = cuda_status(cudaMemcpyAsync(b.h_cur, h_cur, n * row, cudaMemcpyHostToDevice, s));
        if (st == TEE_OK)
            st = cuda_status(cudaMemcpyAsync(b.pos, pos, n * sizeof(int32_t), cudaMemcpyHostToDevice, s));
        if (st == TEE_OK && use_seq)
            st = cuda_status(cudaMemcpyAsync(b.seq, seq, n * sizeof(int32_t), cudaMemcpyHostToDevice, s));
    }
    if (st != TEE_OK) return st;
    // the front (exiting token r scattered to row r of out), then the fill of the
    // exiting tokens at their cache positions (their count stays on the device)
    st = tee_exit_gate_compact_scatter(&step->gate, n, b.h_cur, d, b.h_prev, d, nullptr, nullptr, nullptr, nullptr,
                                       nullptr, nullptr, b.score, b.mask, b.flag, b.cont_rows, b.exit_rows, b.cont_pos,
                                       b.exit_pos, b.h_cont, d, b.out, d, b.n_out, b.counts, b.ws, b.ws_bytes, stream);
    if (st != TEE_OK) return st;
    if (n > 0 && step->n_layers > 0) {
        st = tee_kv_fill(&step->fill, step->n_layers, step->layers, step->prep, step->prep_bytes, n, b.counts + 1,
                         b.h_cur, d, n, b.exit_rows, b.pos, 0, seq && b.seq ? b.seq : nullptr, step->k_cache,
                         step->v_cache, &step->cache, b.ws, b.ws_bytes, stream);
        if (st != TEE_OK) return st;
    }
    // results
    if (mapped) {
        CopyList l{};
        if (score)
            l.seg[l.n++] = CopySeg{reinterpret_cast<const uint8_t*>(b.score), static_cast<uint8_t*>(const_cast<void*>(hv[4])),
                                   static_cast<int64_t>(n * sizeof(float))};
        if (mask)
            l.seg[l.n++] = CopySeg{b.mask, static_cast<uint8_t*>(const_cast<void*>(hv[5])), static_cast<int64_t>(n)};
        if (counts)
            l.seg[l.n++] = CopySeg{reinterpret_cast<const uint8_t*>(b.counts), static_cast<uint8_t*>(const_cast<void*>(hv[6])),
                                   static_cast<int64_t>(2 * sizeof(int32_t))};
        if (out)
            l.seg[l.n++] = CopySeg{static_cast<const uint8_t*>(b.out), static_cast<uint8_t*>(const_cast<void*>(hv[7])),
                                   static_cast<int64_t>(b.n_out) * static_cast<int64_t>(row)};
        return launch_copies(l, true, s);   // a dependent of the fill (or the front)
    }
    if (score) st = cuda_status(cudaMemcpyAsync(score, b.score, n * sizeof(float), cudaMemcpyDeviceToHost, s));
    if (st == TEE_OK && mask) st = cuda_status(cudaMemcpyAsync(mask, b.mask, n, cudaMemcpyDeviceToHost, s));
    if (st == TEE_OK && counts)
        st = cuda_status(cudaMemcpyAsync(counts, b.counts, 2 * sizeof(int32_t), cudaMemcpyDeviceToHost, s));
    if (st == TEE_OK && out)
        st = cuda_status(cudaMemcpyAsync(out, b.out, static_cast<size_t>(b.n_out) * row, cudaMemcpyDeviceToHost, s));
    return st;
}

// Capture the sequence for these arguments into step->exec; false when the runtime
// refuses the capture (the caller then enqueues directly).
bool capture_step(tee_decode_step* step, int n, const void* const (&ptr)[8]) {
    if (step->exec) {
        cudaGraphExecDestroy(step->exec);
        step->exec = nullptr;
    }
    step->g_n = -1;
    const HostViews views = host_views(ptr);
    if (cudaStreamBeginCapture(step->cap, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    const tee_status st = enqueue_step(step, n, ptr[0], ptr[1], static_cast<const int32_t*>(ptr[2]),
                                       static_cast<const int32_t*>(ptr[3]), static_cast<float*>(const_cast<void*>(ptr[4])),
                                       static_cast<uint8_t*>(const_cast<void*>(ptr[5])),
                                       static_cast<int32_t*>(const_cast<void*>(ptr[6])), const_cast<void*>(ptr[7]),
                                       views, step->cap);
    cudaGraph_t graph = nullptr;
    const cudaError_t e = cudaStreamEndCapture(step->cap, &graph);
    bool ok = st == TEE_OK && e == cudaSuccess && graph &&
              cudaGraphInstantiate(&step->exec, graph, 0) == cudaSuccess;
    if (graph) cudaGraphDestroy(graph);
    if (!ok) {
        (void)cudaGetLastError();
        step->exec = nullptr;
        return false;
    }
    step->g_n = n;
    for (int i = 0; i < 8; ++i) step->g_ptr[i] = ptr[i];
    return true;
}

}  // namespace

extern "C" tee_status tee_decode_step_run_host(tee_decode_step* step, int32_t n, const void* h_prev, const void* h_cur,
                                               const int32_t* pos, const int32_t* seq, float* score, uint8_t* mask,
                                               int32_t* counts, void* out, void* stream) {
    if (!step || n < 0 || n > step->n_max || !h_prev || !h_cur || !pos) return TEE_ERR_INVALID_ARG;
    cudaStream_t user = static_cast<cudaStream_t>(stream);
    const void* const ptr[8] = {h_prev, h_cur, pos, seq, score, mask, counts, out};
    bool same = step->exec && step->g_n == n;
    for (int i = 0; i < 8 && same; ++i) same = step->g_ptr[i] == ptr[i];
    if (!same && !step->graph_refused && !capture_step(step, n, ptr)) step->graph_refused = true;
    if (!step->exec || (!same && step->graph_refused))   // no graph for these arguments: enqueue directly
        return enqueue_step(step, n, h_prev, h_cur, pos, seq, score, mask, counts, out, host_views(ptr), user);
    tee_status st = cuda_status(cudaEventRecord(step->ev_in, user));
    if (st == TEE_OK) st = cuda_status(cudaStreamWaitEvent(step->cap, step->ev_in, 0));
    if (st == TEE_OK) st = cuda_status(cudaGraphLaunch(step->exec, step->cap));
    if (st == TEE_OK) st = cuda_status(cudaEventRecord(step->ev_out, step->cap));
    if (st == TEE_OK) st = cuda_status(cudaStreamWaitEvent(user, step->ev_out, 0));
    return st;
}

extern "C" void tee_decode_step_destroy(tee_decode_step* step) {
    if (!step) return;
    if (step->exec) cudaGraphExecDestroy(step->exec);
    if (step->ev_in) cudaEventDestroy(step->ev_in);
    if (step->ev_out) cudaEventDestroy(step->ev_out);
    if (step->cap) cudaStreamDestroy(step->cap);
    delete[] step->layers;
    delete step;
}
