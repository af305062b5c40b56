/*
 * tee.h - token early exit on one GPU: exit gate, compaction, exit scatter and
 * KV fill, as a plain C ABI (libtee.so, built for sm_103a).
 *
 * The four operations follow three write-ups of token-level early exit in
 * decoder-only LLM inference:
 *   - "River-LLM: Large Language Model Seamless Exit Based on KV Share"
 *     (state-transition cosine gate, batch-min rule, KV-shared exit layers
 *     with W4A16 weights that write the skipped layers' cache slots);
 *   - "TIDE: Token-Informed Depth Execution for Per-Token Early Exit in LLM
 *     Inference" (RMSNorm -> router MLP -> sigmoid gate, batch compaction
 *     by warp ballot / prefix sum, exit scatter, exit projection);
 *   - "RidgeFill: training-free later-layer cache fill" (per-layer linear map
 *     from the split state to each later layer's input; that layer's own
 *     norm and K/V projection write the cache).
 *
 * Conventions shared by every call
 *   Ownership: the caller allocates every buffer (device memory unless stated)
 *     and keeps it alive until the work on `stream` has finished. The library
 *     allocates no device memory inside a call.
 *   Streams: `stream` is a cudaStream_t passed as void* (NULL = legacy
 *     default stream). All calls are asynchronous: a call only enqueues
 *     kernels on `stream`, and no call synchronises the host except
 *     tee_get_device_error. Counts stay on the device, so gate -> compact ->
 *     fill -> scatter needs no host round trip.
 *   Layouts: matrices are row-major with a leading dimension `ld` in
 *     elements; device pointers of activations and weights must be 16-byte
 *     aligned and `ld * element size` a multiple of 16 bytes (the kernels use
 *     128-bit loads), and `d` a multiple of 8.
 *   Workspace: each call takes a device scratch buffer `ws` of at least the
 *     size its *_workspace_size query returns. It begins with a 256-byte
 *     header holding a sticky device error word and the counters of the
 *     kernels' "last block" reductions, which every call leaves at zero. The
 *     caller zero-fills a new workspace once (tee_workspace_init); every call
 *     leaves it reusable. A call that stopped on a wait time-out
 *     (TEE_DEVERR_TIMEOUT) may leave a counter set: tee_clear_device_error
 *     zeroes the whole header again. Calls that share one workspace must not
 *     overlap on the GPU.
 *   Errors: every call returns a tee_status. Host-side checks (null required
 *     pointer, bad size, misalignment, unsupported format) return before any
 *     launch. Faults that only the device can see (a row, position, sequence
 *     or destination index out of range) skip the offending write and record
 *     the first such fault in the workspace header; tee_get_device_error
 *     reads it. No kernel traps, and no kernel waits without an iteration
 *     limit.
 */
#ifndef TEE_H
#define TEE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TEE_API __attribute__((visibility("default")))
#else
#define TEE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TEE_OK = 0,
    TEE_ERR_INVALID_ARG = 1,   /* null required pointer, bad size, misaligned pointer or ld, NaN threshold */
    TEE_ERR_UNSUPPORTED = 2,   /* dtype / format combination not built */
    TEE_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed; see tee_last_cuda_error */
    TEE_ERR_WORKSPACE = 4,     /* ws (or prep) missing or smaller than its size query */
    TEE_ERR_DEVICE = 5         /* returned by tee_get_device_error when a device fault was recorded */
} tee_status;

/* Element types. */
enum { TEE_F32 = 0, TEE_F16 = 1, TEE_BF16 = 2 };
/* Gate kinds and exit rules. */
enum { TEE_GATE_COSINE = 0, TEE_GATE_ROUTER = 1 };
enum { TEE_RULE_PER_TOKEN = 0, TEE_RULE_BATCH_ALL = 1 };
/* Weight formats of the fill's K/V projection. */
enum { TEE_W_DENSE = 0, TEE_W_INT4 = 1 };
/* Device fault codes recorded in the workspace header. */
enum {
    TEE_DEVERR_NONE = 0,
    TEE_DEVERR_ROW = 1,        /* a row index outside the source rows */
    TEE_DEVERR_POS = 2,        /* a cache position outside [0, max_pos) */
    TEE_DEVERR_SEQ = 3,        /* a cache sequence outside [0, n_seq) */
    TEE_DEVERR_COUNT = 4,      /* a device-side count larger than its host-side bound */
    TEE_DEVERR_DEST = 5,       /* a scatter destination outside [0, n_out) */
    TEE_DEVERR_TIMEOUT = 6,    /* a pipeline wait ran out of time; the kernel stopped early (detail: where) */
    TEE_DEVERR_NOT_SPD = 7     /* the ridge fit met a pivot <= 0 (detail: the column); the map is NaN */
};

#define TEE_WS_HEADER_BYTES 256

/* ------------------------------------------------------------------ misc */

TEE_API const char* tee_version(void);
TEE_API const char* tee_status_string(tee_status s);
/* The cudaError_t (as int) behind the last TEE_ERR_CUDA of this thread. */
TEE_API int tee_last_cuda_error(void);
/* Zero-fill `bytes` of a workspace on `stream` (needed once per new workspace). */
TEE_API tee_status tee_workspace_init(void* ws, size_t bytes, void* stream);
/* Synchronise `stream`, then report the first device fault recorded in `ws`:
 * *code gets a TEE_DEVERR_* value, *detail the offending index (either may be
 * NULL). Returns TEE_ERR_DEVICE if a fault was recorded, else TEE_OK. */
TEE_API tee_status tee_get_device_error(const void* ws, int32_t* code, int32_t* detail, void* stream);
/* Clear the device fault word of `ws` on `stream`, and every counter of the
 * header with it (the whole TEE_WS_HEADER_BYTES). */
TEE_API tee_status tee_clear_device_error(void* ws, void* stream);

/*
 * Self-check of the failure-detection path: one block of 64 threads waits on an
 * mbarrier that nothing completes, the same bounded wait every pipeline of the
 * library uses, with a limit of limit_us microseconds (1 .. 100000). The waits
 * give up, TEE_DEVERR_TIMEOUT with detail 99 is recorded in the workspace header
 * (read it with tee_get_device_error) and the kernel returns: no fault, no hang,
 * the context stays usable. TEE_ERR_INVALID_ARG for a limit outside the range.
 */
TEE_API tee_status tee_check_wait_timeout(void* ws, uint32_t limit_us, void* stream);
/* Number of kernels this library has launched in this process (all threads). */
TEE_API uint64_t tee_launch_count(void);

/* ------------------------------------------------------------- exit gate */

typedef struct {
    int32_t mode;        /* TEE_GATE_COSINE or TEE_GATE_ROUTER */
    int32_t rule;        /* TEE_RULE_PER_TOKEN or TEE_RULE_BATCH_ALL */
    int32_t dtype;       /* element type of h_cur, h_prev, gamma, w_down, w_up */
    int32_t d;           /* hidden size */
    int32_t bottleneck;  /* router width b (128 in TIDE, at most 256); ignored by the cosine gate */
    float threshold;     /* tau (cosine) or theta (router); exit iff score > threshold */
    float eps;           /* RMSNorm epsilon of the router */
} tee_gate_desc;

/* Workspace for tee_exit_gate: the size at which the router's tensor-core path
 * splits d across the most CTAs. The call also accepts less, down to the size
 * its single-split path needs (about n * 516 bytes + 4 KiB at b = 128); below
 * that it returns TEE_ERR_WORKSPACE. */
TEE_API size_t tee_exit_gate_workspace_size(const tee_gate_desc* desc, int32_t n);

/*
 * Exit gate for n tokens (one row each).
 *
 * Cosine (River-LLM, background "state transition similarity" and method
 * step 3): score[t] = <h_prev[t], h_cur[t]> / (|h_prev[t]| |h_cur[t]|), the
 * similarity of one decoder block's input and output; a zero row scores 0.
 * Router (TIDE, formula 3 and module 4 "Fused LayerNorm + Route"):
 * score[t] = sigmoid(w_up . SiLU(w_down . (g * h_cur[t] / rms(h_cur[t])) +
 * b_down) + b_up), rms(x) = sqrt(mean(x^2) + eps).
 *
 * Rule TEE_RULE_PER_TOKEN: mask[t] = score[t] > threshold. Rule
 * TEE_RULE_BATCH_ALL (River-LLM's min over the batch > tau; TIDE module 3's
 * "for all tokens in the batch"): every mask[t] = (min_t score[t] > threshold).
 * batch_flag (nullable) gets that all-tokens flag under either rule; it is 0
 * for n = 0. Scores accumulate in fp32 and the comparison is taken in fp32.
 *
 *   h_cur   [n][ld_cur]  dtype                    (the block output / router input)
 *   h_prev  [n][ld_prev] dtype                    (cosine only, else NULL)
 *   gamma   [d] dtype, nullable (= 1)             (router only)
 *   w_down  [bottleneck][d] dtype                 (router only)
 *   b_down  [bottleneck] f32, nullable (= 0)      (router only)
 *   w_up    [bottleneck] dtype                    (router only)
 *   b_up    [1] f32, nullable (= 0)               (router only)
 *   score   [n] f32 out;  mask [n] u8 out (1 = exit);  batch_flag [1] i32 out
 */
TEE_API tee_status tee_exit_gate(const tee_gate_desc* desc, int32_t n,
                         const void* h_cur, int64_t ld_cur,
                         const void* h_prev, int64_t ld_prev,
                         const void* gamma, const void* w_down, const float* b_down,
                         const void* w_up, const float* b_up,
                         float* score, uint8_t* mask, int32_t* batch_flag,
                         void* ws, size_t ws_bytes, void* stream);

/*
 * Router gate that needs no workspace (no counterpart on the source pages; it
 * exists for callers that cannot provide device scratch).
 *
 * Meant for callers that cannot allocate device memory when they call the
 * gate: for example a plugin whose host owns all device memory through its
 * own pool and passes in only the call's inputs and outputs, or a
 * latency-critical loop where cudaMalloc is not allowed because it can block
 * or synchronise the device. It computes exactly what tee_exit_gate computes
 * in router mode (same kernels, same arguments without h_prev and without a
 * workspace; the tensor-core path splits d across fewer CTAs when the array is
 * smaller than the size it would ask for), taking its scratch from a 4 MiB array compiled into the
 * library; every GPU that loads the library keeps that array until the
 * process exits. The call itself allocates nothing.
 *
 * Limit: the call is rejected with TEE_ERR_WORKSPACE when the smallest scratch
 * it can run with (see tee_exit_gate_workspace_size) exceeds
 * tee_exit_gate_router_static_max_bytes() (4 MiB), i.e. for more than about
 * 8,000 tokens at bottleneck 128; desc->mode must be TEE_GATE_ROUTER.
 * Set-up: the first call on each device (the device current on the calling
 * thread) looks up the array's device address; make that first call before
 * any stream capture. Sharing: all calls on a device use the same array and
 * it keeps the previous call's contents (each call clears the part that must
 * start at zero), so two calls that overlap on the GPU, on different streams
 * or threads, race and may return wrong results.
 * Faults: a fault only the device sees (a bounded wait of the tensor-core
 * kernel that ran out: TEE_DEVERR_TIMEOUT) is recorded in the array's own
 * fault word, which tee_get_device_error cannot reach. It is sticky: calls do
 * not clear it. Read it with tee_exit_gate_router_static_device_error and
 * clear it with tee_exit_gate_router_static_clear_error.
 */
TEE_API size_t tee_exit_gate_router_static_max_bytes(void);
TEE_API tee_status tee_exit_gate_router_static(const tee_gate_desc* desc, int32_t n,
                                               const void* h, int64_t ld,
                                               const void* gamma, const void* w_down, const float* b_down,
                                               const void* w_up, const float* b_up,
                                               float* score, uint8_t* mask, int32_t* batch_flag,
                                               void* stream);

/*
 * The first device fault recorded by tee_exit_gate_router_static on the
 * current device since the last clear (no counterpart on the source pages).
 * Waits for `stream`, then stores the fault code (TEE_DEVERR_*, 0 if none) and
 * its detail in *code and *detail (either may be NULL). Returns TEE_OK when no
 * fault is recorded, TEE_ERR_DEVICE when one is, TEE_ERR_CUDA on a CUDA error.
 * Like the gate itself, the first use on a device looks up the array's
 * address (before any stream capture).
 */
TEE_API tee_status tee_exit_gate_router_static_device_error(int32_t* code, int32_t* detail, void* stream);

/*
 * Clears the fault word of tee_exit_gate_router_static's array on the current
 * device (an asynchronous write on `stream`); no counterpart on the pages.
 */
TEE_API tee_status tee_exit_gate_router_static_clear_error(void* stream);

/* -------------------------------------------------------- exit compaction */

TEE_API size_t tee_exit_compact_workspace_size(int32_t n);

/*
 * Stable split of n tokens into continuing (mask 0) and exiting (mask != 0)
 * ones (TIDE module 4 "Batch Compact": warp ballot for small batches, a
 * prefix-sum scatter for large ones).
 *
 *   mask      [n] u8 in
 *   pos_in    [n] i32 in, nullable (= row index): original slot of each row
 *   cont_rows [n] i32 out: the first counts[0] entries are the continuing
 *             rows in increasing order; exit_rows likewise for the exiting
 *             rows (first counts[1] entries). Entries past the count are not
 *             written.
 *   cont_pos, exit_pos [n] i32 out, nullable: pos_in of those rows
 *   counts    [2] i32 out (device): {n_cont, n_exit}
 *   h_in      [n][ld_in] dtype, nullable: when given, the continuing rows are
 *             gathered into h_cont [n_cont][ld_cont] (the compacted buffer the
 *             next layer runs on).
 */
TEE_API tee_status tee_exit_compact(int32_t n, const uint8_t* mask, const int32_t* pos_in,
                            const void* h_in, int64_t ld_in, int32_t d, int32_t dtype,
                            int32_t* cont_rows, int32_t* exit_rows,
                            int32_t* cont_pos, int32_t* exit_pos,
                            void* h_cont, int64_t ld_cont, int32_t* counts,
                            void* ws, size_t ws_bytes, void* stream);

/*
 * Compaction and exit scatter in one launch: tee_exit_compact (same arguments
 * and results; the gather into h_cont is optional here, h_cont nullable) and,
 * for every exiting row r, out[p] = h_in[r] with p = pos_in ? pos_in[r] : r,
 * i.e. what tee_exit_scatter(n, counts, exit_rows, exit_pos, h_in, ...) writes
 * without final_gamma. The blocks that rank the rows also copy them, so a
 * decode step saves a launch.
 *
 *   h_in      [n][ld_in] dtype, required
 *   out       [n_out][ld_out] dtype, required; rows other than the exiting
 *             rows' slots are left as they are
 * A slot outside [0, n_out) is skipped and recorded (TEE_DEVERR_DEST).
 * Workspace: tee_exit_compact_workspace_size(n).
 */
TEE_API tee_status tee_exit_compact_scatter(int32_t n, const uint8_t* mask, const int32_t* pos_in,
                            const void* h_in, int64_t ld_in, int32_t d, int32_t dtype,
                            int32_t* cont_rows, int32_t* exit_rows,
                            int32_t* cont_pos, int32_t* exit_pos,
                            void* h_cont, int64_t ld_cont,
                            void* out, int64_t ld_out, int64_t n_out, int32_t* counts,
                            void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------- gate, compaction and scatter */

TEE_API size_t tee_exit_gate_compact_scatter_workspace_size(const tee_gate_desc* desc, int32_t n);

/*
 * The front of a decode step: tee_exit_gate, then tee_exit_compact_scatter on
 * its mask with h = h_cur (continuing rows gathered into h_cont when it is not
 * null, exiting rows scattered to out[pos_in[r] or r]). Arguments and results
 * are those of the two calls. A cosine gate over 1..128 tokens runs as one
 * cluster launch that reads each row once (River-LLM's state-transition cosine
 * with its batch minimum, TIDE module 4's compaction and exit scatter); other
 * calls run the two calls' kernels in turn. out and h_cont must not overlap
 * h_cur. Workspace: tee_exit_gate_compact_scatter_workspace_size.
 */
TEE_API tee_status tee_exit_gate_compact_scatter(const tee_gate_desc* desc, int32_t n,
                            const void* h_cur, int64_t ld_cur,
                            const void* h_prev, int64_t ld_prev,
                            const void* gamma, const void* w_down, const float* b_down,
                            const void* w_up, const float* b_up,
                            const int32_t* pos_in,
                            float* score, uint8_t* mask, int32_t* batch_flag,
                            int32_t* cont_rows, int32_t* exit_rows,
                            int32_t* cont_pos, int32_t* exit_pos,
                            void* h_cont, int64_t ld_cont,
                            void* out, int64_t ld_out, int64_t n_out, int32_t* counts,
                            void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------ exit scatter */

TEE_API size_t tee_exit_scatter_workspace_size(int32_t n_max);

/*
 * Exit scatter (TIDE module 4): for i < counts[1],
 * out[exit_pos[i]] = h_src[exit_rows[i]]; with final_gamma (the "Exit
 * Projection" kernel, RMSNorm fused with the scatter) the row is written as
 * h / sqrt(mean(h^2) + eps) * final_gamma instead. Other rows of `out` are
 * left as they are.
 *
 *   n_max     host bound on counts[1] and on the rows of h_src
 *   counts    [2] i32 device; counts[1] = number of exiting rows
 *   exit_rows, exit_pos [n_max] i32; h_src [n_max][ld_src]; out [n_out][ld_out]
 *   final_gamma [d] dtype, nullable
 * A destination outside [0, n_out) or a source row outside [0, n_max) is
 * skipped and recorded (TEE_DEVERR_DEST / TEE_DEVERR_ROW).
 */
TEE_API tee_status tee_exit_scatter(int32_t n_max, const int32_t* counts,
                            const int32_t* exit_rows, const int32_t* exit_pos,
                            const void* h_src, int64_t ld_src,
                            void* out, int64_t ld_out, int64_t n_out,
                            int32_t d, int32_t dtype, const void* final_gamma, float eps,
                            void* ws, size_t ws_bytes, void* stream);

/* ----------------------------------------------------------------- KV fill */

typedef struct {
    int32_t d;            /* hidden size */
    int32_t n_kv_heads;   /* KV heads written per layer */
    int32_t head_dim;     /* width of one head (even) */
    float rope_base;      /* RoPE base */
    float eps;            /* epsilon of each filled layer's RMSNorm */
    int32_t dtype;        /* h_split, w_map, gamma, dense wk/wv and the caches */
    int32_t wfmt;         /* TEE_W_DENSE or TEE_W_INT4 for wk/wv */
    int32_t group;        /* int4 group length along d (multiple of 16) */
    int32_t flags;        /* 0, or TEE_FILL_EARLY_WEIGHTS and/or TEE_FILL_GENERIC */
} tee_fill_desc;

/* tee_fill_desc.flags. TEE_FILL_EARLY_WEIGHTS: the decode kernel may start while
 * the kernel enqueued just before it on the stream is still running, and read
 * the layers' weights (wk, wv, scales, zeros, gamma) and `prep` at once; it
 * reads h_split, rows, pos, seq, n_dev, the caches and the workspace only after
 * that kernel has completed (programmatic dependent launch). Set it only when
 * that kernel does not write the weights. Ignored by the other paths. */
#define TEE_FILL_EARLY_WEIGHTS 1
/* tee_fill_desc.flags. TEE_FILL_GENERIC: run the call on the generic CUDA-core
 * kernels (a GEMM, RMS and RoPE/store launch per step and layer) even where a
 * fused path (tensor-core prefill, int4 decode, small dense one-launch fill)
 * takes it; same results within rounding. For checking one path against
 * another. */
#define TEE_FILL_GENERIC 2

/* Weights of one filled layer j (device pointers). kvw = n_kv_heads*head_dim. */
typedef struct {
    const void* w_map;    /* [d][d] dtype: x_j = h_split . w_map; NULL = identity (state propagation) */
    const void* gamma;    /* [d] dtype: layer j's RMSNorm weight */
    const void* wk;       /* dense [d][kvw] dtype, or int4 [d/2][kvw] u8 (even k in the low nibble) */
    const void* wv;       /* same as wk */
    const void* k_scale;  /* int4 only: [d/group][kvw] f16; W = (q - zero) * scale */
    const void* k_zero;   /* int4 only: [d/group][kvw] f16 */
    const void* v_scale;
    const void* v_zero;
    int32_t cache_layer;  /* layer index into the caches */
    int32_t writes;       /* caches this layer writes: 0 (both), TEE_FILL_WRITE_K, TEE_FILL_WRITE_V */
    /* Model-family variants (RidgeFill's per-model notes); all nullable:
     * k = x^ Wk + k_bias, v = x^ Wv + v_bias (QKV-bias models); with k_norm,
     * each head of k is RMS-normalised over head_dim (eps = desc->eps) and
     * multiplied by k_norm before RoPE (QK-norm models). dtype of h. */
    const void* k_bias;   /* [kvw] */
    const void* v_bias;   /* [kvw] */
    const void* k_norm;   /* [head_dim] */
} tee_fill_layer;

/* tee_fill_layer.writes: fill only the K cache (V kept as the backbone wrote
 * it) or only the V cache: RidgeFill finds the fill's error in K on one model
 * family and in V on another. */
#define TEE_FILL_WRITE_K 1
#define TEE_FILL_WRITE_V 2

/* Cache geometry, shared by k_cache and v_cache. Strides are in elements;
 * head_dim is contiguous. Slot (layer, seq, head, pos) starts at
 * layer*s_layer + seq*s_seq + head*s_head + pos*s_pos and holds head_dim
 * elements. n_heads must be at least the descriptor's n_kv_heads. */
typedef struct {
    int64_t s_layer, s_seq, s_head, s_pos;
    int32_t n_layers, n_seq, n_heads, max_pos;
} tee_cache_layout;

/* Size of the prepared-state buffer `prep` (RoPE table and repacked weights). */
TEE_API size_t tee_kv_fill_prep_size(const tee_fill_desc* desc, int32_t n_layers, int32_t max_pos);
/* Fill `prep` for these layers and positions [0, max_pos). Run once, and again
 * whenever the weights behind `layers` change; tee_kv_fill reads it. */
TEE_API tee_status tee_kv_fill_prepare(const tee_fill_desc* desc, int32_t n_layers, const tee_fill_layer* layers,
                               int32_t max_pos, void* prep, size_t prep_bytes, void* stream);

TEE_API size_t tee_kv_fill_workspace_size(const tee_fill_desc* desc, int32_t n_layers, int32_t n_max);

/*
 * KV fill for the layers an exiting token skips.
 *
 * RidgeFill: x_j = h_split . W_j, the split-layer state mapped to filled
 * layer j's input by a per-layer ridge map (identity = River-LLM's State
 * Propagation); then layer j's own RMSNorm x^ = x_j / rms(x_j) * gamma_j and
 * projections k = x^ . Wk_j, v = x^ . Wv_j (dense, or River-LLM's W4A16 int4
 * weights); RoPE (rotate-half pairs i, i + head_dim/2, angle
 * pos * rope_base^(-2i/head_dim)) on each K head; K and V stored in the slot
 * the backbone would have written (River-LLM method step 1: identical
 * position index, head split and dimension layout).
 *
 * Items: n = *n_dev if n_dev is given (a device count, e.g. counts + 1 of
 * tee_exit_compact), else n_max; n must not exceed n_max. Item i uses
 *   row r = rows ? rows[i] : i            of h_split (r < h_rows),
 *   position p = pos ? pos[r] : pos0 + r  (0 <= p < cache->max_pos),
 *   sequence s = seq ? seq[r] : 0         (0 <= s < cache->n_seq),
 * and writes every kv head of every listed layer.
 *
 *   layers     host array of n_layers descriptors (device weight pointers)
 *   prep       prepared by tee_kv_fill_prepare for the same desc and layers
 *   h_split    [h_rows][ld_h] dtype
 *   k_cache, v_cache  caches of `dtype` laid out as `cache` says
 */
TEE_API tee_status tee_kv_fill(const tee_fill_desc* desc, int32_t n_layers, const tee_fill_layer* layers,
                       const void* prep, size_t prep_bytes,
                       int32_t n_max, const int32_t* n_dev,
                       const void* h_split, int64_t ld_h, int32_t h_rows,
                       const int32_t* rows, const int32_t* pos, int32_t pos0, const int32_t* seq,
                       void* k_cache, void* v_cache, const tee_cache_layout* cache,
                       void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------- ridge fit (next) */

TEE_API size_t tee_ridge_fit_workspace_size(int32_t n, int32_t d, int32_t d_out);

/*
 * RidgeFill's per-layer map, fitted on the GPU (RidgeFill, "closed-form ridge
 * regression" note): W = (X^T X + lambda I)^-1 X^T Y over n calibration rows.
 *
 *   x     [n][ld_x] bf16: split-layer states;  y [n][ld_y] bf16: the true
 *         inputs of the filled layer
 *   w     [d][ld_w] f32 out: the map, for x_j = h W (tee_kv_fill's w_map
 *         after a conversion to the fill's dtype)
 *   d, d_out multiples of 256; lambda >= 0
 * X^T X and X^T Y accumulate in fp32 on the tensor cores; the Cholesky
 * factorisation and the two triangular solves run in fp32. A pivot <= 0
 * (X^T X + lambda I not positive definite in fp32) records
 * TEE_DEVERR_NOT_SPD and leaves NaN in w.
 */
TEE_API tee_status tee_ridge_fit(int32_t n, int32_t d, int32_t d_out, const void* x, int64_t ld_x,
                                 const void* y, int64_t ld_y, int32_t dtype, float lambda,
                                 float* w, int64_t ld_w, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------ Exit River (next) */

/* One int4 weight matrix W [k_in][n_out] in the fill's W4A16 format: codes
 * [k_in/2][n_out] u8 (two per byte along k, even k in the low nibble), f16
 * scale and zero [k_in/group][n_out]; W = (q - zero) * scale. */
typedef struct {
    const void* codes;
    const void* scale;
    const void* zero;
} tee_w4;

typedef struct {
    int32_t d;            /* hidden size (multiple of 128) */
    int32_t n_q_heads;    /* query heads (a multiple of n_kv_heads) */
    int32_t n_kv_heads;   /* KV heads */
    int32_t head_dim;     /* 64 or 128 */
    int32_t d_ff;         /* FFN width (multiple of 64) */
    float rope_base;      /* RoPE base (q and k) */
    float eps;            /* epsilon of both RMSNorms */
    int32_t group;        /* int4 group length: 64 */
    int32_t flags;        /* 0, or one of TEE_RIVER_ATTN_BY_PAIR / TEE_RIVER_ATTN_BY_CHUNK */
} tee_river_desc;

/* tee_river_desc.flags: how the attention walks the cache; same results within
 * rounding. By default it walks whole (item, kv head) pairs, one persistent
 * consumer group per pair with an online softmax over the pair's chunks, when
 * n_max * n_kv_heads fills every group (two per SM) or the cache is too long for
 * the other walk's merge (above ~87 K positions at head_dim 64 with 8 query
 * heads per kv head), and otherwise splits each sequence into chunks of one CTA
 * each whose partial results a merge combines (its workspace then holds the
 * partials: it grows with max_pos). These force one walk; the workspace size
 * follows the flag, and the chunk walk on a cache too long for it returns
 * TEE_ERR_UNSUPPORTED. */
#define TEE_RIVER_ATTN_BY_PAIR 1
#define TEE_RIVER_ATTN_BY_CHUNK 2

/* One exit layer: the W4A16 copy of decoder layer `cache_layer` (device
 * pointers). qw = n_q_heads*head_dim, kvw = n_kv_heads*head_dim. */
typedef struct {
    const void* attn_norm;  /* [d] bf16: RMSNorm weight before attention */
    const void* ffn_norm;   /* [d] bf16: RMSNorm weight before the FFN */
    tee_w4 wq;              /* [d][qw] */
    tee_w4 wk;              /* [d][kvw] */
    tee_w4 wv;              /* [d][kvw] */
    tee_w4 wo;              /* [qw][d] */
    tee_w4 wg;              /* [d][d_ff] gate */
    tee_w4 wu;              /* [d][d_ff] up */
    tee_w4 wd;              /* [d_ff][d] down */
    int32_t cache_layer;    /* layer index into the caches */
    int32_t reserved;       /* 0 */
} tee_river_layer;

/* Size of `prep`: the layers' weights repacked per 128-column tile (each k
 * block's codes, scales and zeros contiguous; about 1.1x the int4 weights) and
 * the RoPE table for positions [0, max_pos). */
TEE_API size_t tee_exit_river_prep_size(const tee_river_desc* desc, int32_t n_layers, int32_t max_pos);
/* Fill `prep` for these layers (run again whenever their weights change);
 * tee_exit_river reads it with the same desc and the same layers in order. */
TEE_API tee_status tee_exit_river_prepare(const tee_river_desc* desc, int32_t n_layers,
                                          const tee_river_layer* layers, int32_t max_pos, void* prep,
                                          size_t prep_bytes, void* stream);
/* Workspace of a call with up to n_max items over caches of cache->max_pos
 * positions. */
TEE_API size_t tee_exit_river_workspace_size(const tee_river_desc* desc, int32_t n_max, int32_t max_pos);

/*
 * River-LLM's Exit River (core method; method steps 1 and 3): the tokens that
 * left the backbone continue through the W4A16 copies of the remaining
 * layers, each of which writes the skipped layer's K/V into the backbone's
 * own slots and passes its output to the next; the last output goes to the
 * LM head. Per exit layer, for every item:
 *   x = RMSNorm(h) * attn_norm;  q, k, v = x Wq, x Wk, x Wv;
 *   RoPE (rotate-half, as tee_kv_fill) on every head of q and k at the item's
 *   position; k, v stored at (cache_layer, seq, head, pos) -- every item's
 *   before any attention of the layer;
 *   o_h = softmax(q_h . K^T / sqrt(head_dim)) . V over positions 0..pos of the
 *   item's sequence, q head h reading kv head h / (n_q_heads / n_kv_heads);
 *   h1 = h + o . Wo;  x2 = RMSNorm(h1) * ffn_norm;
 *   h <- h1 + (SiLU(x2 Wg) * (x2 Wu)) . Wd.
 * The residual stream stays in fp32 between layers; contractions take bf16
 * operands (int4 weights dequantised to bf16) and accumulate in fp32.
 *
 * Items: n = *n_dev if n_dev is given, else n_max (n_max <= 128). Item i uses
 *   row r = rows ? rows[i] : i of h (r < h_rows), position pos[r] and
 *   sequence seq ? seq[r] : 0, and writes h_out[i] (item order, ready for
 *   tee_exit_scatter). An item with a bad row, position or sequence is
 *   recorded (TEE_DEVERR_ROW / POS / SEQ) and skipped: no cache write, and
 *   h_out[i] is left as it was.
 *
 *   layers     host array of n_layers exit layers, in order
 *   prep       prepared by tee_exit_river_prepare for the same desc and layers
 *              (the weights are read from there; the layers' weight pointers
 *              are not read by this call)
 *   h          [h_rows][ld_h] bf16;  h_out [n_max][ld_out] bf16
 *   k_cache, v_cache  bf16 caches laid out as `cache` says
 */
TEE_API tee_status tee_exit_river(const tee_river_desc* desc, int32_t n_layers, const tee_river_layer* layers,
                                  const void* prep, size_t prep_bytes, int32_t n_max, const int32_t* n_dev,
                                  const void* h, int64_t ld_h, int32_t h_rows, const int32_t* rows,
                                  const int32_t* pos, const int32_t* seq,
                                  void* k_cache, void* v_cache, const tee_cache_layout* cache,
                                  void* h_out, int64_t ld_out, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------- decode step from host buffers */

/*
 * One whole decode step, host memory to host memory, in one call: River-LLM's
 * exit decision and KV fill (method steps 1 and 3) with TIDE module 4's
 * compaction and exit scatter. The call copies the step's inputs from host
 * memory into the device buffers the step was created with, runs
 * tee_exit_gate_compact_scatter (gate, compaction with the continuing rows
 * gathered, exit scatter of token r into row r of `out`), then tee_kv_fill for
 * the exiting tokens at their cache positions
 * (rows = exit_rows, item count = counts[1] on the device, h_split = h_cur),
 * and copies the score, the mask, the counts and `out` back to host memory;
 * everything is enqueued on `stream` and the host results are valid once the
 * stream has completed. Host buffers should be page-locked for the copies to
 * run asynchronously; when every one is page-locked memory that the device
 * reaches directly, two copy kernels move them (all inputs in one launch, all
 * results in another) instead of one cudaMemcpyAsync per buffer. The results equal those of the two calls made on the
 * device buffers. The step object captures the sequence into a CUDA graph on a
 * stream of its own at the first call and replays it while n and the host
 * pointers stay the same (events order it after and before `stream`); with
 * pageable host memory, where the capture is refused, it enqueues the calls on
 * `stream` directly. One step object must not be run from two threads at once.
 */
typedef struct {
    /* device buffers owned by the caller, alive as long as the step object */
    void* h_prev;          /* [n_max][d] gate dtype: the previous layer's states */
    void* h_cur;           /* [n_max][d] gate dtype: the current layer's states (and the fill's h_split) */
    int32_t* pos;          /* [n_max] cache position of each token */
    int32_t* seq;          /* [n_max] cache sequence of each token; NULL = sequence 0 */
    float* score;          /* [n_max] */
    uint8_t* mask;         /* [n_max] */
    int32_t* flag;         /* [1] batch flag, or NULL */
    int32_t* cont_rows;    /* [n_max] */
    int32_t* exit_rows;    /* [n_max] */
    int32_t* cont_pos;     /* [n_max] or NULL */
    int32_t* exit_pos;     /* [n_max] or NULL */
    void* h_cont;          /* [n_max][d] or NULL: the continuing rows gathered */
    void* out;             /* [n_out][d]: exiting token r's row scattered to out[r] (n_out >= n_max) */
    int64_t n_out;
    int32_t* counts;       /* [2] continuing, exiting */
    void* ws;              /* workspace for both calls */
    size_t ws_bytes;
} tee_step_buffers;

typedef struct tee_decode_step tee_decode_step;   /* opaque; host memory only */

/* Check and keep the descriptors, the fill's layers (copied), its prepared
 * state, the caches and the buffers. gate->mode must be TEE_GATE_COSINE; the
 * gate's d and dtype must match the fill's. Errors: TEE_ERR_INVALID_ARG for a
 * null or inconsistent argument, TEE_ERR_WORKSPACE when buf->ws is smaller
 * than both calls need at n_max. *step is set only on success. */
TEE_API tee_status tee_decode_step_create(const tee_gate_desc* gate, int32_t n_max, const tee_fill_desc* fill,
                                          int32_t n_layers, const tee_fill_layer* layers, const void* fill_prep,
                                          size_t fill_prep_bytes, void* k_cache, void* v_cache,
                                          const tee_cache_layout* cache, const tee_step_buffers* buf,
                                          tee_decode_step** step);

/* One step over n <= n_max tokens. Host inputs: h_prev, h_cur [n][d] (gate
 * dtype, rows contiguous), pos [n], seq [n] or NULL. Host outputs (each may be
 * NULL to skip its copy): score [n], mask [n], counts [2], out [n_out][d]. */
TEE_API tee_status tee_decode_step_run_host(tee_decode_step* step, int32_t n, const void* h_prev, const void* h_cur,
                                            const int32_t* pos, const int32_t* seq, float* score, uint8_t* mask,
                                            int32_t* counts, void* out, void* stream);

/* Free the step object (not the buffers it was given). NULL is allowed. */
TEE_API void tee_decode_step_destroy(tee_decode_step* step);

#ifdef __cplusplus
}
#endif
#endif /* TEE_H */
