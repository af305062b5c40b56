// Batch compaction and exit scatter (TIDE core module 4).
//
// Compaction is a stable split of the batch rows by the exit mask. Each block
// owns a chunk of R rows (R = 32..256). Inside the chunk every warp takes 32
// rows and ranks them with one __ballot_sync + __popc (the warp-ballot path;
// a batch of at most 32 tokens is exactly one warp). Across chunks the
// offsets are a prefix sum of exit counts: for batches up to PREFIX_DIRECT_MAX
// rows each block counts the exits before its chunk straight from the mask
// bytes (a few KB, read from L2), so the whole split is one launch with no
// inter-block waiting; larger batches first write per-chunk counts to the
// workspace and each block sums the counts before it. The same blocks then
// gather their continuing rows into the compacted buffer with 128-bit copies.
//
// The exit scatter copies each exiting row back to its original slot; with a
// final RMSNorm weight it is TIDE's "Exit Projection" (norm fused with scatter).
// Without that norm the scatter can also run inside the compaction launch: the
// blocks that rank the rows copy their exiting rows to `out` beside the gather of
// the continuing rows (one launch fewer on a decode step).
#include "common.cuh"

namespace tee {

namespace {

constexpr int CP_THREADS = 256;
constexpr int CP_WARPS = CP_THREADS / 32;
constexpr int PREFIX_DIRECT_MAX = 1 << 16;

// Number of non-zero bytes in a 32-bit word.
__device__ __forceinline__ unsigned nonzero_bytes(uint32_t w) {
    const uint32_t t = ((w & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | w;
    return __popc(t & 0x80808080u);
}

// Exits among mask[0, end), counted by the whole block (result on every thread).
__device__ unsigned block_count_exits(const uint8_t* __restrict__ mask, int end, unsigned* s_red) {
    unsigned c = 0;
    const uintptr_t base = reinterpret_cast<uintptr_t>(mask);
    const int mis = static_cast<int>((16 - (base & 15)) & 15);
    const int head = mis < end ? mis : end;
    for (int i = threadIdx.x; i < head; i += CP_THREADS) c += mask[i] != 0;
    const int nvec = (end - head) / 16;
    const uint4* v = reinterpret_cast<const uint4*>(mask + head);
    for (int i = threadIdx.x; i < nvec; i += CP_THREADS) {
        const uint4 u = v[i];
        c += nonzero_bytes(u.x) + nonzero_bytes(u.y) + nonzero_bytes(u.z) + nonzero_bytes(u.w);
    }
    for (int i = head + nvec * 16 + threadIdx.x; i < end; i += CP_THREADS) c += mask[i] != 0;
    c = warp_sum_u(c);
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = c;
    __syncthreads();
    unsigned tot = 0;
#pragma unroll
    for (int w = 0; w < CP_WARPS; ++w) tot += s_red[w];
    __syncthreads();
    return tot;
}

// Pass 1 of the large-batch path: exits per chunk.
__global__ void __launch_bounds__(CP_THREADS)
chunk_count_kernel(int n, int R, const uint8_t* __restrict__ mask, uint32_t* __restrict__ chunk_exits) {
    __shared__ unsigned s_red[CP_WARPS];
    const int r0 = blockIdx.x * R;
    unsigned c = 0;
    for (int i = r0 + threadIdx.x; i < min(r0 + R, n); i += CP_THREADS) c += mask[i] != 0;
    c = warp_sum_u(c);
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = c;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned tot = 0;
        for (int w = 0; w < CP_WARPS; ++w) tot += s_red[w];
        chunk_exits[blockIdx.x] = tot;
    }
}

template <typename T>
__global__ void __launch_bounds__(CP_THREADS)
compact_kernel(int n, int R, const uint8_t* __restrict__ mask, const int32_t* __restrict__ pos_in,
               const uint32_t* __restrict__ chunk_exits, const T* __restrict__ h_in, int64_t ld_in, int d,
               int32_t* __restrict__ cont_rows, int32_t* __restrict__ exit_rows, int32_t* __restrict__ cont_pos,
               int32_t* __restrict__ exit_pos, T* __restrict__ h_cont, int64_t ld_cont,
               int32_t* __restrict__ counts, T* __restrict__ out, int64_t ld_out, int64_t n_out, void* ws) {
    allow_dependents();
    __shared__ unsigned s_red[CP_WARPS];
    __shared__ unsigned s_wexit[CP_WARPS];
    __shared__ int s_src[256];     // the chunk's continuing rows, in order
    __shared__ int s_xsrc[256];    // its exiting rows, in order, and their slots in `out`
    __shared__ int s_xdst[256];
    const int r0 = blockIdx.x * R;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // Exits before this chunk.
    unsigned prefix;
    if (chunk_exits) {
        unsigned c = 0;
        for (int i = threadIdx.x; i < static_cast<int>(blockIdx.x); i += CP_THREADS) c += chunk_exits[i];
        c = warp_sum_u(c);
        if (lane == 0) s_red[warp] = c;
        __syncthreads();
        prefix = 0;
#pragma unroll
        for (int w = 0; w < CP_WARPS; ++w) prefix += s_red[w];
        __syncthreads();
    } else {
        prefix = block_count_exits(mask, r0, s_red);
    }

    // Warp ballots inside the chunk (R may be below 32: lanes past it sit out).
    const int row = r0 + warp * 32 + lane;
    const bool active = warp * 32 < R;
    const bool in = active && warp * 32 + lane < R && row < n;
    const bool is_exit = in && mask[row] != 0;
    const unsigned ball = __ballot_sync(0xFFFFFFFFu, is_exit);
    if (lane == 0) s_wexit[warp] = active ? __popc(ball) : 0u;
    __syncthreads();
    unsigned before = prefix;
    unsigned chunk_total = 0;
#pragma unroll
    for (int w = 0; w < CP_WARPS; ++w) {
        if (w < warp) before += s_wexit[w];
        chunk_total += s_wexit[w];
    }
    if (in) {
        const unsigned lt = __popc(ball & ((1u << lane) - 1u));
        const int e_idx = static_cast<int>(before + lt);      // exits before this row
        const int c_idx = row - e_idx;                          // continuing rows before it
        const int32_t p = pos_in ? pos_in[row] : row;
        const int local = c_idx - (r0 - static_cast<int>(prefix));  // continuing rows of this chunk before it
        if (is_exit) {
            if (e_idx >= 0 && e_idx < n) {
                exit_rows[e_idx] = row;
                if (exit_pos) exit_pos[e_idx] = p;
            }
            const int xl = e_idx - static_cast<int>(prefix);   // exiting rows of this chunk before it
            if (xl >= 0 && xl < 256) {
                s_xsrc[xl] = row;
                s_xdst[xl] = p;
            }
        } else if (c_idx >= 0 && c_idx < n && local >= 0 && local < 256) {
            cont_rows[c_idx] = row;
            if (cont_pos) cont_pos[c_idx] = p;
            s_src[local] = row;
        }
    }
    const int chunk_rows = min(R, n - r0);
    if (r0 + chunk_rows == n && threadIdx.x == 0) {
        const int n_exit = static_cast<int>(prefix + chunk_total);
        counts[0] = n - n_exit;
        counts[1] = n_exit;
    }
    if (!h_in) return;
    __syncthreads();
    // Copy the chunk's rows, one warp per row, 16 bytes per lane: the continuing
    // rows into h_cont (gather), then the exiting rows to their slots of `out`
    // (scatter), in one sequence of jobs over the block's warps.
    const int n_cont_chunk = h_cont ? min(chunk_rows - static_cast<int>(chunk_total), R) : 0;
    const int n_exit_chunk = out ? min(static_cast<int>(chunk_total), R) : 0;
    const int dst0 = r0 - static_cast<int>(prefix);
    constexpr int V = 16 / sizeof(T);
    for (int j = warp; j < n_cont_chunk + n_exit_chunk; j += CP_WARPS) {
        if (j < n_cont_chunk) {
            const uint4* src = reinterpret_cast<const uint4*>(h_in + static_cast<int64_t>(s_src[j]) * ld_in);
            uint4* dst = reinterpret_cast<uint4*>(h_cont + static_cast<int64_t>(dst0 + j) * ld_cont);
            warp_copy16(dst, src, d / V, lane);
        } else {
            const int x = j - n_cont_chunk;
            const int64_t slot = s_xdst[x];
            if (slot < 0 || slot >= n_out) {
                if (lane == 0) record_fault(ws, TEE_DEVERR_DEST, static_cast<int>(slot));
                continue;
            }
            const uint4* src = reinterpret_cast<const uint4*>(h_in + static_cast<int64_t>(s_xsrc[x]) * ld_in);
            warp_copy16(reinterpret_cast<uint4*>(out + slot * ld_out), src, d / V, lane);
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(256)
scatter_kernel(int n_max, const int32_t* __restrict__ counts, const int32_t* __restrict__ exit_rows,
               const int32_t* __restrict__ exit_pos, const T* __restrict__ h_src, int64_t ld_src,
               T* __restrict__ out, int64_t ld_out, int64_t n_out, int d, const T* __restrict__ gamma, float eps,
               void* ws) {
    allow_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // The row lists hold n_max entries: read this warp's first entries together with
    // the count instead of after it (one dependent load fewer on the critical path).
    const int i_first = blockIdx.x * 8 + warp;
    const int src_first = i_first < n_max ? exit_rows[i_first] : 0;
    const int64_t dst_first = i_first < n_max ? exit_pos[i_first] : 0;
    int n_exit = counts[1];
    if (n_exit > n_max) {
        if (blockIdx.x == 0 && threadIdx.x == 0) record_fault(ws, TEE_DEVERR_COUNT, n_exit);
        n_exit = n_max;
    }
    for (int i = i_first; i < n_exit; i += gridDim.x * 8) {
        const int src = i == i_first ? src_first : exit_rows[i];
        const int64_t dst = i == i_first ? dst_first : exit_pos[i];
        if (src < 0 || src >= n_max) {
            if (lane == 0) record_fault(ws, TEE_DEVERR_ROW, src);
            continue;
        }
        if (dst < 0 || dst >= n_out) {
            if (lane == 0) record_fault(ws, TEE_DEVERR_DEST, static_cast<int>(dst));
            continue;
        }
        const T* s = h_src + static_cast<int64_t>(src) * ld_src;
        T* o = out + dst * ld_out;
        if (!gamma) {
            constexpr int V = 16 / sizeof(T);
            warp_copy16(reinterpret_cast<uint4*>(o), reinterpret_cast<const uint4*>(s), d / V, lane);
            continue;
        }
        float ss = 0.f;
        for (int k = lane * 8; k < d; k += 256) {
            float x[8];
            load8(s + k, x);
#pragma unroll
            for (int q = 0; q < 8; ++q) ss = fmaf(x[q], x[q], ss);
        }
        ss = warp_sum(ss);
        const float r = 1.0f / sqrtf(ss / static_cast<float>(d) + eps);
        for (int k = lane * 8; k < d; k += 256) {
            float x[8], g[8];
            load8(s + k, x);
            load8(gamma + k, g);
#pragma unroll
            for (int q = 0; q < 8; ++q) x[q] = x[q] * r * g[q];
            store8(o + k, x);
        }
    }
}

// Rows per block: about one block per SM. Calls that copy rows start from 8 rows a
// block (one row per warp), so that a small batch's copies spread over SMs.
int chunk_rows_for(int n, bool copies) {
    if (n > PREFIX_DIRECT_MAX) return 256;
    const int target = copies ? (n + 147) / 148 : (n + 147) / 148 * 4;
    int R = copies ? 8 : 32;
    while (R < target && R < 256) R <<= 1;
    return R;
}

template <typename T>
tee_status run_compact(int n, const uint8_t* mask, const int32_t* pos_in, const void* h_in, int64_t ld_in, int d,
                       int32_t* cont_rows, int32_t* exit_rows, int32_t* cont_pos, int32_t* exit_pos, void* h_cont,
                       int64_t ld_cont, int32_t* counts, void* out, int64_t ld_out, int64_t n_out, void* ws,
                       cudaStream_t s) {
    const int R = chunk_rows_for(n, h_in != nullptr);
    const int chunks = (n + R - 1) / R;
    uint32_t* chunk_exits = nullptr;
    if (n > PREFIX_DIRECT_MAX) {
        chunk_exits = ws_at<uint32_t>(ws, TEE_WS_HEADER_BYTES);
        chunk_count_kernel<<<chunks, CP_THREADS, 0, s>>>(n, R, mask, chunk_exits);
        tee_status st = launch_status();
        if (st != TEE_OK) return st;
    }
    compact_kernel<T><<<chunks, CP_THREADS, 0, s>>>(n, R, mask, pos_in, chunk_exits, static_cast<const T*>(h_in),
                                                    ld_in, d, cont_rows, exit_rows, cont_pos, exit_pos,
                                                    static_cast<T*>(h_cont), ld_cont, counts, static_cast<T*>(out),
                                                    ld_out, n_out, ws);
    return launch_status();
}

}  // namespace

}  // namespace tee

using namespace tee;

extern "C" size_t tee_exit_compact_workspace_size(int32_t n) {
    if (n < 0) return 0;
    return TEE_WS_HEADER_BYTES + (n > PREFIX_DIRECT_MAX ? round_up((static_cast<size_t>(n) + 255) / 256 * 4, 256) : 0);
}

static tee_status compact_call(int32_t n, const uint8_t* mask, const int32_t* pos_in, const void* h_in,
                               int64_t ld_in, int32_t d, int32_t dtype, int32_t* cont_rows, int32_t* exit_rows,
                               int32_t* cont_pos, int32_t* exit_pos, void* h_cont, int64_t ld_cont, void* out,
                               int64_t ld_out, int64_t n_out, int32_t* counts, void* ws, size_t ws_bytes,
                               void* stream) {
    if (n < 0 || !counts) return TEE_ERR_INVALID_ARG;
    if (!ws || ws_bytes < tee_exit_compact_workspace_size(n)) return TEE_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (n == 0) return cuda_status(cudaMemsetAsync(counts, 0, 2 * sizeof(int32_t), s));
    if (!mask || !cont_rows || !exit_rows) return TEE_ERR_INVALID_ARG;
    if (h_in) {
        const size_t es = dtype_bytes(dtype);
        if (es == 0) return TEE_ERR_UNSUPPORTED;
        if ((!h_cont && !out) || d <= 0 || (d * es) % 16 || ld_in < d || (ld_in * es) % 16 || !aligned16(h_in))
            return TEE_ERR_INVALID_ARG;
        if (h_cont && (ld_cont < d || (ld_cont * es) % 16 || !aligned16(h_cont))) return TEE_ERR_INVALID_ARG;
        if (out && (n_out < 0 || ld_out < d || (ld_out * es) % 16 || !aligned16(out))) return TEE_ERR_INVALID_ARG;
    }
    switch (h_in ? dtype : TEE_BF16) {
        case TEE_F32:
            return run_compact<float>(n, mask, pos_in, h_in, ld_in, d, cont_rows, exit_rows, cont_pos, exit_pos,
                                      h_cont, ld_cont, counts, out, ld_out, n_out, ws, s);
        case TEE_F16:
            return run_compact<__half>(n, mask, pos_in, h_in, ld_in, d, cont_rows, exit_rows, cont_pos, exit_pos,
                                       h_cont, ld_cont, counts, out, ld_out, n_out, ws, s);
        default:
            return run_compact<__nv_bfloat16>(n, mask, pos_in, h_in, ld_in, d, cont_rows, exit_rows, cont_pos,
                                              exit_pos, h_cont, ld_cont, counts, out, ld_out, n_out, ws, s);
    }
}

extern "C" tee_status tee_exit_compact(int32_t n, const uint8_t* mask, const int32_t* pos_in, const void* h_in,
                                       int64_t ld_in, int32_t d, int32_t dtype, int32_t* cont_rows,
                                       int32_t* exit_rows, int32_t* cont_pos, int32_t* exit_pos, void* h_cont,
                                       int64_t ld_cont, int32_t* counts, void* ws, size_t ws_bytes, void* stream) {
    if (h_in && !h_cont) return TEE_ERR_INVALID_ARG;
    return compact_call(n, mask, pos_in, h_in, ld_in, d, dtype, cont_rows, exit_rows, cont_pos, exit_pos, h_cont,
                        ld_cont, nullptr, 0, 0, counts, ws, ws_bytes, stream);
}

extern "C" tee_status tee_exit_compact_scatter(int32_t n, const uint8_t* mask, const int32_t* pos_in,
                                               const void* h_in, int64_t ld_in, int32_t d, int32_t dtype,
                                               int32_t* cont_rows, int32_t* exit_rows, int32_t* cont_pos,
                                               int32_t* exit_pos, void* h_cont, int64_t ld_cont, void* out,
                                               int64_t ld_out, int64_t n_out, int32_t* counts, void* ws,
                                               size_t ws_bytes, void* stream) {
    if (n > 0 && (!h_in || !out)) return TEE_ERR_INVALID_ARG;
    return compact_call(n, mask, pos_in, h_in, ld_in, d, dtype, cont_rows, exit_rows, cont_pos, exit_pos, h_cont,
                        ld_cont, out, ld_out, n_out, counts, ws, ws_bytes, stream);
}

extern "C" size_t tee_exit_scatter_workspace_size(int32_t n_max) {
    (void)n_max;
    return TEE_WS_HEADER_BYTES;
}

extern "C" tee_status tee_exit_scatter(int32_t n_max, const int32_t* counts, const int32_t* exit_rows,
                                       const int32_t* exit_pos, const void* h_src, int64_t ld_src, void* out,
                                       int64_t ld_out, int64_t n_out, int32_t d, int32_t dtype,
                                       const void* final_gamma, float eps, void* ws, size_t ws_bytes,
                                       void* stream) {
    if (n_max < 0 || n_out < 0) return TEE_ERR_INVALID_ARG;
    if (!ws || ws_bytes < tee_exit_scatter_workspace_size(n_max)) return TEE_ERR_WORKSPACE;
    if (n_max == 0) return TEE_OK;
    const size_t es = dtype_bytes(dtype);
    if (es == 0) return TEE_ERR_UNSUPPORTED;
    if (!counts || !exit_rows || !exit_pos || !h_src || !out || d <= 0 || d % 8 || ld_src < d || ld_out < d ||
        (ld_src * es) % 16 || (ld_out * es) % 16 || !aligned16(h_src) || !aligned16(out))
        return TEE_ERR_INVALID_ARG;
    if (final_gamma && (!aligned16(final_gamma) || !(eps >= 0.f))) return TEE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int blocks = (n_max + 7) / 8;
    const int cap = sm_count() * 8;
    if (blocks > cap) blocks = cap;
    switch (dtype) {
        case TEE_F32:
            scatter_kernel<float><<<blocks, 256, 0, s>>>(n_max, counts, exit_rows, exit_pos,
                                                         static_cast<const float*>(h_src), ld_src,
                                                         static_cast<float*>(out), ld_out, n_out, d,
                                                         static_cast<const float*>(final_gamma), eps, ws);
            break;
        case TEE_F16:
            scatter_kernel<__half><<<blocks, 256, 0, s>>>(n_max, counts, exit_rows, exit_pos,
                                                          static_cast<const __half*>(h_src), ld_src,
                                                          static_cast<__half*>(out), ld_out, n_out, d,
                                                          static_cast<const __half*>(final_gamma), eps, ws);
            break;
        default:
            scatter_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(
                n_max, counts, exit_rows, exit_pos, static_cast<const __nv_bfloat16*>(h_src), ld_src,
                static_cast<__nv_bfloat16*>(out), ld_out, n_out, d, static_cast<const __nv_bfloat16*>(final_gamma),
                eps, ws);
            break;
    }
    return launch_status();
}
