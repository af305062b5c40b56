// KV fill for the layers an exiting token skips.
//
// RidgeFill (idea source section): the split-layer state h is mapped to each
// later layer's input x_j = h W_j; that layer's own RMSNorm and K/V
// projection then write the cache as the backbone would. With W_j = I this is
// River-LLM's State Propagation. River-LLM (method step 1) keeps the exit
// layer's cache addressing identical to the backbone and stores its weights
// as W4A16 (4-bit weights, 16-bit activations).
//
// This file holds the prepared state (RoPE table, computed in float64 so that
// positions up to ~10^6 keep their angle to ~1e-7 rad), the workspace layout,
// the entry points, and the generic CUDA-core path that handles every
// dtype / format / row-gather combination. Large bf16 fills with dense weights
// go to the tensor-core path (fill_tc.cu); small int4 decode fills to the
// decode path (fill_decode.cu).
#include "fill.cuh"

namespace tee {

namespace {

// ------------------------------------------------------------ RoPE table
__global__ void rope_table_kernel(int max_pos, int half, double base, float2* __restrict__ table) {
    const int64_t total = static_cast<int64_t>(max_pos) * half;
    for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int p = static_cast<int>(idx / half);
        const int i = static_cast<int>(idx % half);
        const double inv_freq = pow(base, -2.0 * i / (2.0 * half));
        const double ang = static_cast<double>(p) * inv_freq;
        double s, c;
        sincos(ang, &s, &c);
        table[idx] = make_float2(static_cast<float>(c), static_cast<float>(s));
    }
}

// ------------------------------------------------------------ generic path
constexpr int GB_M = 64, GB_N = 64, GB_K = 16, GB_THREADS = 256;

// Row source of the A operand: either gathered rows of h_split (dtype T) or
// the fp32 map output X held in the workspace.
template <typename T>
struct ARows {
    const T* h;            // h_split, used when x == nullptr
    int64_t ld_h;
    const int32_t* rows;   // nullable
    int h_rows;
    const float* x;        // fp32 [n_max][d] map output, nullable
    const T* colscale;     // gamma, nullable
    const float* rowscale; // 1/rms per item, nullable
};

// B operand: columns [0, nsplit) come from b0, [nsplit, N) from b1.
template <typename T>
struct BCols {
    const void* b0;
    const void* b1;
    int nsplit;
    int ldb;               // columns of each source
    int int4;              // 1: packed int4 with fp16 scale/zero
    const __half* s0; const __half* z0; const __half* s1; const __half* z1;
    int group;
};

template <typename T>
__device__ __forceinline__ float load_b(const BCols<T>& B, int k, int c) {
    const bool second = c >= B.nsplit;
    const int cc = second ? c - B.nsplit : c;
    if (!B.int4) {
        const T* src = static_cast<const T*>(second ? B.b1 : B.b0);
        return to_f32(src[static_cast<int64_t>(k) * B.ldb + cc]);
    }
    const uint8_t* src = static_cast<const uint8_t*>(second ? B.b1 : B.b0);
    const uint8_t byte = src[static_cast<int64_t>(k >> 1) * B.ldb + cc];
    const float q = static_cast<float>((k & 1) ? (byte >> 4) : (byte & 15));
    const int64_t gi = static_cast<int64_t>(k / B.group) * B.ldb + cc;
    const float s = __half2float((second ? B.s1 : B.s0)[gi]);
    const float z = __half2float((second ? B.z1 : B.z0)[gi]);
    return (q - z) * s;
}

// C[m][c] = sum_k A(m,k) * B(k,c), fp32 accumulate, for m < item count.
template <typename T>
__global__ void __launch_bounds__(GB_THREADS)
generic_gemm_kernel(int n_max, const int32_t* __restrict__ n_dev, int K, int N, ARows<T> A, BCols<T> B,
                    float* __restrict__ C, int64_t ldc, void* ws) {
    const int n = item_count(n_max, n_dev);
    const int m0 = blockIdx.y * GB_M, c0 = blockIdx.x * GB_N;
    if (m0 >= n) return;
    __shared__ float As[GB_K][GB_M + 4];
    __shared__ float Bs[GB_K][GB_N + 4];
    const int tid = threadIdx.x;
    const int tx = tid % 16, ty = tid / 16;
    // A loader: row am, k offsets ak..ak+3
    const int am = tid / 4, ak = (tid % 4) * 4;
    const int m = m0 + am;
    int src_row = -1;
    if (m < n) {
        src_row = A.rows ? A.rows[m] : m;
        if (!A.x && (src_row < 0 || src_row >= A.h_rows)) {
            if (ak == 0) record_fault(ws, TEE_DEVERR_ROW, src_row);
            src_row = -1;
        }
    }
    const float rs = (m < n && A.rowscale) ? A.rowscale[m] : 1.f;
    const int bk = tid / 16, bc = (tid % 16) * 4;
    float acc[4][4] = {};
    // The next k tile is loaded into registers while the current one is multiplied
    // from shared memory, so that a k step does not wait for its loads.
    float ra[4], rb[4];
    auto load_tile = [&](int k0) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int k = k0 + ak + q;
            float v = 0.f;
            if (src_row >= 0 && k < K) {
                v = A.x ? A.x[static_cast<int64_t>(m) * K + k] : to_f32(A.h[static_cast<int64_t>(src_row) * A.ld_h + k]);
                if (A.colscale) v *= to_f32(A.colscale[k]);
                v *= rs;
            }
            ra[q] = v;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int k = k0 + bk, c = c0 + bc + q;
            rb[q] = (k < K && c < N) ? load_b(B, k, c) : 0.f;
        }
    };
    load_tile(0);
    for (int k0 = 0; k0 < K; k0 += GB_K) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            As[ak + q][am] = ra[q];
            Bs[bk][bc + q] = rb[q];
        }
        __syncthreads();
        if (k0 + GB_K < K) load_tile(k0 + GB_K);
#pragma unroll
        for (int kk = 0; kk < GB_K; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int mm = m0 + ty * 4 + i;
        if (mm >= n) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int c = c0 + tx * 4 + j;
            if (c < N) C[static_cast<int64_t>(mm) * ldc + c] = acc[i][j];
        }
    }
}

// rowscale[m] = 1 / sqrt(mean(x_m^2) + eps) where x_m is X[m] or h_split[row(m)].
template <typename T>
__global__ void __launch_bounds__(256)
generic_rms_kernel(int n_max, const int32_t* __restrict__ n_dev, int d, float eps, ARows<T> A,
                   float* __restrict__ rowscale) {
    const int n = item_count(n_max, n_dev);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m = blockIdx.x * 8 + warp;
    if (m >= n) return;
    float ss = 0.f;
    if (A.x) {
        const float* x = A.x + static_cast<int64_t>(m) * d;
        for (int k = lane; k < d; k += 32) ss = fmaf(x[k], x[k], ss);
    } else {
        const int r = A.rows ? A.rows[m] : m;
        if (r >= 0 && r < A.h_rows) {
            const T* x = A.h + static_cast<int64_t>(r) * A.ld_h;
            for (int k = lane; k < d; k += 32) {
                const float v = to_f32(x[k]);
                ss = fmaf(v, v, ss);
            }
        }
    }
    ss = warp_sum(ss);
    if (lane == 0) rowscale[m] = 1.0f / sqrtf(ss / static_cast<float>(d) + eps);
}

// Bias, the optional per-head K norm, RoPE on K, and the store of K and V into
// the backbone's slots: a warp per (item, kv head), lanes over the rotation pairs.
template <typename T>
__global__ void __launch_bounds__(256)
generic_rope_store_kernel(int n_max, const int32_t* __restrict__ n_dev, int n_kv, int hd, const float* __restrict__ kv,
                          int h_rows, const int32_t* __restrict__ rows, const int32_t* __restrict__ pos, int pos0,
                          const int32_t* __restrict__ seq, const PrepHeader* __restrict__ hdr,
                          const float2* __restrict__ rope, T* __restrict__ kc, T* __restrict__ vc,
                          tee_cache_layout cl, int layer, const T* __restrict__ kb, const T* __restrict__ vb,
                          const T* __restrict__ kn, float eps, int writes, void* ws) {
    const int n = item_count(n_max, n_dev);
    const int half = hd / 2, kvw = n_kv * hd;
    const int lane = threadIdx.x & 31;
    const bool write_k = writes != TEE_FILL_WRITE_V, write_v = writes != TEE_FILL_WRITE_K;
    const int64_t total = static_cast<int64_t>(n) * n_kv;
    for (int64_t w = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5; w < total;
         w += (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5) {
        const int m = static_cast<int>(w / n_kv), h = static_cast<int>(w % n_kv);
        const int r = rows ? rows[m] : m;
        if (r < 0 || r >= h_rows) continue;  // recorded by the GEMM's row check
        const int p = pos ? pos[r] : pos0 + r;
        const int s = seq ? seq[r] : 0;
        if (!pos_ok(p, cl.max_pos, hdr)) {
            if (h == 0 && lane == 0) record_fault(ws, TEE_DEVERR_POS, p);
            continue;
        }
        if (s < 0 || s >= cl.n_seq) {
            if (h == 0 && lane == 0) record_fault(ws, TEE_DEVERR_SEQ, s);
            continue;
        }
        const float* row = kv + static_cast<int64_t>(m) * 2 * kvw;
        const int64_t off = layer * cl.s_layer + s * cl.s_seq + h * cl.s_head + static_cast<int64_t>(p) * cl.s_pos;
        // K: bias, then the head's RMS (when normalised) over all hd values
        float krs = 1.f;
        if (kn) {
            float ss = 0.f;
            for (int i = lane; i < hd; i += 32) {
                const float k = row[h * hd + i] + (kb ? to_f32(kb[h * hd + i]) : 0.f);
                ss = fmaf(k, k, ss);
            }
            krs = 1.0f / sqrtf(warp_sum(ss) / static_cast<float>(hd) + eps);
        }
        for (int i = lane; i < half; i += 32) {
            if (write_k) {
                float k1 = row[h * hd + i], k2 = row[h * hd + i + half];
                if (kb) {
                    k1 += to_f32(kb[h * hd + i]);
                    k2 += to_f32(kb[h * hd + i + half]);
                }
                if (kn) {
                    k1 *= krs * to_f32(kn[i]);
                    k2 *= krs * to_f32(kn[i + half]);
                }
                const float2 cs = rope[static_cast<int64_t>(p) * half + i];
                kc[off + i] = from_f32<T>(k1 * cs.x - k2 * cs.y);
                kc[off + i + half] = from_f32<T>(k2 * cs.x + k1 * cs.y);
            }
            if (write_v) {
                float v1 = row[kvw + h * hd + i], v2 = row[kvw + h * hd + i + half];
                if (vb) {
                    v1 += to_f32(vb[h * hd + i]);
                    v2 += to_f32(vb[h * hd + i + half]);
                }
                vc[off + i] = from_f32<T>(v1);
                vc[off + i + half] = from_f32<T>(v2);
            }
        }
    }
}

template <typename T>
tee_status run_generic(const FillCall& fc) {
    const tee_fill_desc& D = *fc.desc;
    const int d = D.d, kvw = D.n_kv_heads * D.head_dim;
    const GenericWs w = generic_ws(D, fc.n_max);
    float* X = ws_at<float>(fc.ws, w.x_off);
    float* rs = ws_at<float>(fc.ws, w.r_off);
    float* KV = ws_at<float>(fc.ws, w.kv_off);
    const PrepView pv = prep_view(fc.prep, D, fc.n_layers);
    for (int l = 0; l < fc.n_layers; ++l) {
        const tee_fill_layer& L = fc.layers[l];
        ARows<T> A{static_cast<const T*>(fc.h), fc.ld_h, fc.rows, fc.h_rows, nullptr, nullptr, nullptr};
        if (L.w_map) {
            BCols<T> B{L.w_map, L.w_map, d, d, 0, nullptr, nullptr, nullptr, nullptr, D.group};
            dim3 grid((d + GB_N - 1) / GB_N, (fc.n_max + GB_M - 1) / GB_M);
            generic_gemm_kernel<T><<<grid, GB_THREADS, 0, fc.stream>>>(fc.n_max, fc.n_dev, d, d, A, B, X, d, fc.ws);
            tee_status st = launch_status();
            if (st != TEE_OK) return st;
            A.x = X;
        }
        generic_rms_kernel<T><<<(fc.n_max + 7) / 8, 256, 0, fc.stream>>>(fc.n_max, fc.n_dev, d, D.eps, A, rs);
        tee_status st = launch_status();
        if (st != TEE_OK) return st;
        A.colscale = static_cast<const T*>(L.gamma);
        A.rowscale = rs;
        BCols<T> B{L.wk, L.wv, kvw, kvw, D.wfmt == TEE_W_INT4,
                   static_cast<const __half*>(L.k_scale), static_cast<const __half*>(L.k_zero),
                   static_cast<const __half*>(L.v_scale), static_cast<const __half*>(L.v_zero), D.group};
        dim3 grid((2 * kvw + GB_N - 1) / GB_N, (fc.n_max + GB_M - 1) / GB_M);
        generic_gemm_kernel<T><<<grid, GB_THREADS, 0, fc.stream>>>(fc.n_max, fc.n_dev, d, 2 * kvw, A, B, KV,
                                                                   2 * kvw, fc.ws);
        st = launch_status();
        if (st != TEE_OK) return st;
        const int64_t warps = static_cast<int64_t>(fc.n_max) * D.n_kv_heads;
        int blocks = static_cast<int>((warps + 7) / 8);
        if (blocks > 4 * 1024) blocks = 4 * 1024;
        if (blocks < 1) blocks = 1;
        generic_rope_store_kernel<T><<<blocks, 256, 0, fc.stream>>>(
            fc.n_max, fc.n_dev, D.n_kv_heads, D.head_dim, KV, fc.h_rows, fc.rows, fc.pos, fc.pos0, fc.seq, pv.hdr, pv.rope,
            static_cast<T*>(fc.k_cache), static_cast<T*>(fc.v_cache), *fc.cache, L.cache_layer,
            static_cast<const T*>(L.k_bias), static_cast<const T*>(L.v_bias), static_cast<const T*>(L.k_norm), D.eps,
            L.writes, fc.ws);
        st = launch_status();
        if (st != TEE_OK) return st;
    }
    return TEE_OK;
}

}  // namespace

GenericWs generic_ws(const tee_fill_desc& D, int n_max) {
    GenericWs w;
    const size_t n = static_cast<size_t>(n_max > 0 ? n_max : 1);
    const size_t kvw = static_cast<size_t>(D.n_kv_heads) * D.head_dim;
    w.x_off = TEE_WS_HEADER_BYTES;
    w.r_off = round_up(w.x_off + n * D.d * 4, 256);
    w.kv_off = round_up(w.r_off + n * 4, 256);
    w.end = round_up(w.kv_off + n * 2 * kvw * 4, 256);
    return w;
}

tee_status build_rope_table(float2* table, int max_pos, int half, double base, cudaStream_t s) {
    const int64_t total = static_cast<int64_t>(max_pos) * half;
    int blocks = static_cast<int>((total + 255) / 256);
    if (blocks > 8192) blocks = 8192;
    if (blocks < 1) blocks = 1;
    rope_table_kernel<<<blocks, 256, 0, s>>>(max_pos, half, base, table);
    return launch_status();
}

}  // namespace tee

using namespace tee;

static tee_status check_fill_desc(const tee_fill_desc* D) {
    if (!D || D->d <= 0 || D->d % 8 || D->n_kv_heads <= 0 || D->head_dim <= 0 || D->head_dim % 8)
        return TEE_ERR_INVALID_ARG;
    if (!(D->rope_base > 1.f) || !(D->eps >= 0.f)) return TEE_ERR_INVALID_ARG;
    if (dtype_bytes(D->dtype) == 0) return TEE_ERR_UNSUPPORTED;
    if (D->wfmt != TEE_W_DENSE && D->wfmt != TEE_W_INT4) return TEE_ERR_UNSUPPORTED;
    if (D->wfmt == TEE_W_INT4 && (D->group <= 0 || D->group % 16 || D->d % D->group)) return TEE_ERR_INVALID_ARG;
    if (D->flags & ~(TEE_FILL_EARLY_WEIGHTS | TEE_FILL_GENERIC)) return TEE_ERR_INVALID_ARG;
    return TEE_OK;
}

extern "C" size_t tee_kv_fill_prep_size(const tee_fill_desc* D, int32_t n_layers, int32_t max_pos) {
    if (check_fill_desc(D) != TEE_OK || n_layers < 0 || max_pos <= 0) return 0;
    return PREP_HEADER_BYTES + fill_tc_prep_bytes(*D, n_layers) + fill_decode_prep_bytes(*D, n_layers) +
           rope_table_bytes(max_pos, D->head_dim);
}

extern "C" tee_status tee_kv_fill_prepare(const tee_fill_desc* D, int32_t n_layers, const tee_fill_layer* layers,
                                          int32_t max_pos, void* prep, size_t prep_bytes, void* stream) {
    tee_status st = check_fill_desc(D);
    if (st != TEE_OK) return st;
    if (n_layers < 0 || max_pos <= 0 || (n_layers > 0 && !layers)) return TEE_ERR_INVALID_ARG;
    if (!prep || !aligned16(prep) || prep_bytes < tee_kv_fill_prep_size(D, n_layers, max_pos)) return TEE_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    PrepHeader h{};
    h.magic = PREP_MAGIC;
    h.d = D->d;
    h.n_kv_heads = D->n_kv_heads;
    h.head_dim = D->head_dim;
    h.max_pos = max_pos;
    h.n_layers = n_layers;
    h.tc_layers = fill_tc_prep_bytes(*D, n_layers) ? n_layers : 0;
    h.dec_layers = fill_decode_prep_bytes(*D, n_layers) ? n_layers : 0;
    // The header copy is staged from pageable memory before cudaMemcpyAsync returns.
    st = cuda_status(cudaMemcpyAsync(prep, &h, sizeof(h), cudaMemcpyHostToDevice, s));
    if (st != TEE_OK) return st;
    const PrepView pv = prep_view(prep, *D, n_layers);
    st = build_rope_table(const_cast<float2*>(pv.rope), max_pos, D->head_dim / 2, D->rope_base, s);
    if (st != TEE_OK) return st;
    st = fill_tc_prepare(*D, n_layers, layers, const_cast<char*>(pv.tc), s);
    if (st != TEE_OK) return st;
    return fill_decode_prepare(*D, n_layers, layers, const_cast<char*>(pv.dec), s);
}

extern "C" size_t tee_kv_fill_workspace_size(const tee_fill_desc* D, int32_t n_layers, int32_t n_max) {
    if (check_fill_desc(D) != TEE_OK || n_max < 0 || n_layers < 0) return 0;
    size_t a = generic_ws(*D, n_max).end;
    size_t b = fill_tc_ws_bytes(*D, n_layers, n_max);
    size_t c = fill_decode_ws_bytes(*D, n_layers, n_max);
    size_t m = a > b ? a : b;
    return m > c ? m : c;
}

extern "C" tee_status tee_kv_fill(const tee_fill_desc* D, int32_t n_layers, const tee_fill_layer* layers,
                                  const void* prep, size_t prep_bytes, int32_t n_max, const int32_t* n_dev,
                                  const void* h_split, int64_t ld_h, int32_t h_rows, const int32_t* rows,
                                  const int32_t* pos, int32_t pos0, const int32_t* seq, void* k_cache, void* v_cache,
                                  const tee_cache_layout* cache, void* ws, size_t ws_bytes, void* stream) {
    tee_status st = check_fill_desc(D);
    if (st != TEE_OK) return st;
    if (n_layers < 0 || n_max < 0 || h_rows < 0 || pos0 < 0) return TEE_ERR_INVALID_ARG;
    if (!ws || ws_bytes < tee_kv_fill_workspace_size(D, n_layers, n_max)) return TEE_ERR_WORKSPACE;
    if (n_layers == 0 || n_max == 0) return TEE_OK;
    if (!layers || !h_split || !k_cache || !v_cache || !cache) return TEE_ERR_INVALID_ARG;
    if (!prep || prep_bytes < tee_kv_fill_prep_size(D, n_layers, cache->max_pos))
        return TEE_ERR_WORKSPACE;
    const size_t es = dtype_bytes(D->dtype);
    if (ld_h < D->d || (ld_h * es) % 16 || !aligned16(h_split)) return TEE_ERR_INVALID_ARG;
    if (!rows && !n_dev && n_max > h_rows) return TEE_ERR_INVALID_ARG;
    if (cache->n_layers <= 0 || cache->n_seq <= 0 || cache->max_pos <= 0 || cache->n_heads < D->n_kv_heads)
        return TEE_ERR_INVALID_ARG;
    if (cache->s_pos < D->head_dim || cache->s_head < D->head_dim || cache->s_seq < 0 || cache->s_layer < 0)
        return TEE_ERR_INVALID_ARG;
    if (!pos && !rows && !n_dev && static_cast<int64_t>(pos0) + n_max > cache->max_pos) return TEE_ERR_INVALID_ARG;
    for (int l = 0; l < n_layers; ++l) {
        const tee_fill_layer& L = layers[l];
        if (!L.gamma || !L.wk || !L.wv || L.cache_layer < 0 || L.cache_layer >= cache->n_layers)
            return TEE_ERR_INVALID_ARG;
        if (D->wfmt == TEE_W_INT4 && (!L.k_scale || !L.k_zero || !L.v_scale || !L.v_zero)) return TEE_ERR_INVALID_ARG;
        if (L.writes != 0 && L.writes != TEE_FILL_WRITE_K && L.writes != TEE_FILL_WRITE_V) return TEE_ERR_INVALID_ARG;
        if ((L.k_bias && !aligned16(L.k_bias)) || (L.v_bias && !aligned16(L.v_bias)) || (L.k_norm && !aligned16(L.k_norm)))
            return TEE_ERR_INVALID_ARG;
    }
    FillCall fc{D, n_layers, layers, prep, prep_bytes, n_max, n_dev, h_split, ld_h, h_rows, rows, pos, pos0, seq,
                k_cache, v_cache, cache, ws, ws_bytes, static_cast<cudaStream_t>(stream)};
    if (!(D->flags & TEE_FILL_GENERIC)) {
        st = fill_tc_run(fc);
        if (st != TEE_ERR_UNSUPPORTED) return st;
        st = fill_decode_run(fc);
        if (st != TEE_ERR_UNSUPPORTED) return st;
        st = fill_small_run(fc);
        if (st != TEE_ERR_UNSUPPORTED) return st;
    }
    switch (D->dtype) {
        case TEE_F32: return run_generic<float>(fc);
        case TEE_F16: return run_generic<__half>(fc);
        default: return run_generic<__nv_bfloat16>(fc);
    }
}
