// Small dense KV fill in one launch (RidgeFill "idea source": the map, the
// filled layer's RMSNorm and its K/V projections; River-LLM method step 1:
// RoPE and the store into the backbone's slot). For decode batches of a few
// items on small models, where the generic path's four launches per layer are
// all latency.
//
// Scope: dense weights in the activation type, n_max <= 32 items, d a multiple
// of 32 up to 2048 with n_max * d <= 16384, head_dim <= 256, at most 64 layers
// per launch (more are launched in groups).
//
// One cluster of 8 CTAs per filled layer; CTA r of the cluster:
//   1. stages the items' h rows as fp32 [n][d] in shared memory (16-byte loads);
//   2. ridge map: computes columns [r d/8, (r+1) d/8) of x = h W_j for every
//      item and the partial sums of x^2 over them; one cluster barrier; reads
//      the eight column slices and partial sums through distributed shared
//      memory and forms x^ = x / rms(x) * gamma_j over the whole row.
//      Identity map: x = h, the sum of squares over the whole row locally.
//   3. takes heads r, r + 8, ... of the layer's 2 n_kv heads (K heads, then V
//      heads) and computes them as in 2 (x^ times the head's columns of Wk or
//      Wv); adds the bias; for K, the optional per-head RMS norm and RoPE from
//      the table; stores the head into the cache slot.
// The products run on CUDA cores with fp32 accumulation: lanes over 32 output
// columns, the eight warps over d, their sums added in shared memory. When they
// fit, the CTA's weight slices (its map columns and its heads' columns of Wk /
// Wv) are copied into shared memory with cp.async at the start -- under an
// early (programmatic) launch, while the previous kernel still runs.
#include "fill.cuh"

namespace tee {

namespace {

constexpr int SF_CLUSTER = 8;
constexpr int SF_THREADS = 256;
constexpr int SF_WARPS = SF_THREADS / 32;
constexpr int SF_MAX_ITEMS = 32;
constexpr int SF_MAX_ELEMS = 16384;   // n_max * d: the staged rows, fp32
constexpr int SF_MAX_D = 2048;
constexpr int SF_MAX_HD = 256;
constexpr int SF_MAX_LAYERS = 64;

struct SmallLayer {
    const void* w_map;     // nullable: identity
    const void* gamma;
    const void* wk;
    const void* wv;
    const void* k_bias;
    const void* v_bias;
    const void* k_norm;
    int cache_layer;
    int writes;
};

struct SmallArgs {
    int n_max;
    const int32_t* n_dev;
    int d, n_kv, hd;
    float eps;
    const void* h;
    int64_t ld_h;
    int h_rows;
    const int32_t* rows;
    const int32_t* pos;
    int pos0;
    const int32_t* seq;
    const PrepHeader* hdr;
    const float2* rope;
    void* k_cache;
    void* v_cache;
    tee_cache_layout cl;
    int early;
    int stage;             // the weight slices are copied into shared memory
    int has_map;           // some layer has a ridge map (the staged map slice exists)
    int n_layers;
    SmallLayer l[SF_MAX_LAYERS];
};

// Shared memory (floats): A [n_max][d] | xs [n_max][d/8] | red [8][NM][32] |
// hv [n_max][hd] | ssp [32] | rs [32]; ints: ok [32], pos [32], off [32] (int64);
// then, when staged, the weight slices (element type T): the map's [d][d/8] and
// per head slot [d][hd] (slot i = the CTA's i-th head, heads r, r + 8, ...).
struct SmallLayout {
    size_t a, xs, red, hv, ssp, rs, ok, p, off, w, bytes, staged_bytes;
};
__host__ __device__ inline int heads_per_cta(int n_kv) { return (2 * n_kv + SF_CLUSTER - 1) / SF_CLUSTER; }
inline __host__ __device__ SmallLayout small_layout(int n_max, int d, int hd, int nm, int n_kv, int es, bool map) {
    SmallLayout s;
    s.a = 0;
    s.xs = s.a + static_cast<size_t>(n_max) * d * 4;
    s.red = s.xs + static_cast<size_t>(n_max) * (d / SF_CLUSTER) * 4;
    s.hv = s.red + static_cast<size_t>(SF_WARPS) * nm * 32 * 4;
    s.ssp = s.hv + static_cast<size_t>(n_max) * hd * 4;
    s.rs = s.ssp + SF_MAX_ITEMS * 4;
    s.ok = s.rs + SF_MAX_ITEMS * 4;
    s.p = s.ok + SF_MAX_ITEMS * 4;
    s.off = (s.p + SF_MAX_ITEMS * 4 + 7) / 8 * 8;
    s.w = (s.off + SF_MAX_ITEMS * 8 + 127) / 128 * 128;
    s.bytes = s.w;
    s.staged_bytes = s.w + (map ? static_cast<size_t>(d) * (d / SF_CLUSTER) * es : 0) +
                     static_cast<size_t>(heads_per_cta(n_kv)) * d * hd * es;
    return s;
}

__device__ __forceinline__ uint32_t sf_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void sf_cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void sf_cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t sf_peer(const float* local, int rank) {
    uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local)), r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}
__device__ __forceinline__ float sf_ld_peer(const float* local, int rank) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(sf_peer(local, rank)) : "memory");
    return v;
}
__device__ __forceinline__ float4 sf_ld_peer4(const float* local, int rank) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(sf_peer(local, rank))
                 : "memory");
    return v;
}

__device__ __forceinline__ void sf_cp16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src)
                 : "memory");
}
// Rows [0, K) x bytes [0, row_bytes) of src (row pitch src_pitch bytes) into dst
// (rows packed), 16 bytes per cp.async, all threads of the CTA.
__device__ __forceinline__ void stage_rows(uint8_t* dst, const uint8_t* src, int K, int row_bytes, int64_t src_pitch) {
    const int per = row_bytes / 16;
    for (int i = threadIdx.x; i < K * per; i += SF_THREADS) {
        const int k = i / per, q = i - k * per;
        sf_cp16(dst + static_cast<size_t>(k) * row_bytes + q * 16, src + k * src_pitch + q * 16);
    }
}

// out[m][oc + j] = sum_{k < K} A[m][k] * B[k][c0 + j] for m < n, j < ncols
// (<= 32), A fp32 [n][lda] in shared memory, B row-major [K][ldb] in global
// memory. Lane j owns column c0 + j; warp w the k range [w K/8, (w+1) K/8),
// four k at a time (K % 32 == 0, lda % 4 == 0). Ends with the block in step.
template <typename T, int NM>
__device__ void col_pass(const float* __restrict__ A, int lda, int n, int K, const T* __restrict__ B, int64_t ldb,
                         int c0, int ncols, float* __restrict__ red, float* __restrict__ out, int ldo, int oc) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool cv = lane < ncols;
    const int kw = K / SF_WARPS;
    const int k_lo = warp * kw;
    const T* bp = B + static_cast<int64_t>(k_lo) * ldb + c0 + (cv ? lane : 0);
    float acc[NM];
#pragma unroll
    for (int m = 0; m < NM; ++m) acc[m] = 0.f;
    // 16 k a batch, every load of the batch issued before its arithmetic (from
    // global memory each batch costs one round trip)
    constexpr int KB = 16;
    for (int k0 = 0; k0 < kw; k0 += KB) {
        float b[KB];
#pragma unroll
        for (int q = 0; q < KB; ++q)
            b[q] = (cv && k0 + q < kw) ? to_f32(bp[static_cast<int64_t>(k0 + q) * ldb]) : 0.f;
#pragma unroll
        for (int q4 = 0; q4 < KB; q4 += 4) {
            if (k0 + q4 >= kw) break;
#pragma unroll
            for (int m = 0; m < NM; ++m) {
                if (m < n) {
                    const float4 a = *reinterpret_cast<const float4*>(A + m * lda + k_lo + k0 + q4);
                    acc[m] = fmaf(a.x, b[q4], acc[m]);
                    acc[m] = fmaf(a.y, b[q4 + 1], acc[m]);
                    acc[m] = fmaf(a.z, b[q4 + 2], acc[m]);
                    acc[m] = fmaf(a.w, b[q4 + 3], acc[m]);
                }
            }
        }
    }
#pragma unroll
    for (int m = 0; m < NM; ++m)
        if (m < n) red[(warp * NM + m) * 32 + lane] = acc[m];
    __syncthreads();
    for (int i = threadIdx.x; i < n * 32; i += SF_THREADS) {
        const int m = i >> 5, j = i & 31;
        if (j < ncols) {
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < SF_WARPS; ++w) s += red[(w * NM + m) * 32 + j];
            out[m * ldo + oc + j] = s;
        }
    }
    __syncthreads();
}

template <typename T, int NM>
__global__ void __cluster_dims__(SF_CLUSTER, 1, 1) __launch_bounds__(SF_THREADS, 1)
fill_small_kernel(const __grid_constant__ SmallArgs a, void* ws) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int d = a.d, hd = a.hd, half = hd / 2, kvw = a.n_kv * hd;
    const int cpc = d / SF_CLUSTER;
    constexpr int es = static_cast<int>(sizeof(T));
    const SmallLayout lay = small_layout(a.n_max, d, hd, NM, a.n_kv, es, a.has_map);
    float* As = reinterpret_cast<float*>(smem + lay.a);
    float* xs = reinterpret_cast<float*>(smem + lay.xs);
    float* red = reinterpret_cast<float*>(smem + lay.red);
    float* hv = reinterpret_cast<float*>(smem + lay.hv);
    float* ssp = reinterpret_cast<float*>(smem + lay.ssp);
    float* rs = reinterpret_cast<float*>(smem + lay.rs);
    int* ok = reinterpret_cast<int*>(smem + lay.ok);
    int* ps = reinterpret_cast<int*>(smem + lay.p);
    int64_t* offs = reinterpret_cast<int64_t*>(smem + lay.off);
    const int rank = static_cast<int>(sf_rank());
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const SmallLayer& L = a.l[blockIdx.y];
    const T* wmap = static_cast<const T*>(L.w_map);
    const T* gamma = static_cast<const T*>(L.gamma);
    const bool write_k = L.writes != TEE_FILL_WRITE_V, write_v = L.writes != TEE_FILL_WRITE_K;

    // Weights do not depend on the previous kernel: they are requested first.
    uint8_t* w_map_s = smem + lay.w;                                            // [d][cpc]
    uint8_t* w_head_s = w_map_s + (a.has_map ? static_cast<size_t>(d) * cpc * es : 0);   // slots of [d][hd]
    if (a.stage) {
        if (wmap)
            stage_rows(w_map_s, reinterpret_cast<const uint8_t*>(wmap + rank * cpc), d, cpc * es,
                       static_cast<int64_t>(d) * es);
        int slot = 0;
        for (int hh = rank; hh < 2 * a.n_kv; hh += SF_CLUSTER, ++slot) {
            const bool is_k = hh < a.n_kv;
            if (is_k ? !write_k : !write_v) continue;
            const T* w = static_cast<const T*>(is_k ? L.wk : L.wv) + (is_k ? hh : hh - a.n_kv) * hd;
            stage_rows(w_head_s + static_cast<size_t>(slot) * d * hd * es, reinterpret_cast<const uint8_t*>(w), d,
                       hd * es, static_cast<int64_t>(kvw) * es);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
        if (a.early) wait_prior_grid();
    } else if (a.early) {
        // pull this CTA's slices into L2 while the previous kernel runs
        if (wmap)
            for (int k = threadIdx.x; k < d; k += SF_THREADS)
                for (int b = 0; b < cpc * es; b += 128)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(
                                     wmap + static_cast<int64_t>(k) * d + rank * cpc) + b));
        for (int hh = rank; hh < 2 * a.n_kv; hh += SF_CLUSTER) {
            const bool is_k = hh < a.n_kv;
            if (is_k ? !write_k : !write_v) continue;
            const T* w = static_cast<const T*>(is_k ? L.wk : L.wv) + (is_k ? hh : hh - a.n_kv) * hd;
            for (int k = threadIdx.x; k < d; k += SF_THREADS)
                for (int b = 0; b < hd * es; b += 128)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(
                                     w + static_cast<int64_t>(k) * kvw) + b));
        }
        wait_prior_grid();
    }
    const int n = item_count(a.n_max, a.n_dev);

    // Items: source row, position, sequence; faults recorded once per layer by rank 0.
    if (threadIdx.x < SF_MAX_ITEMS) {
        const int m = threadIdx.x;
        int good = 0, p = 0;
        int64_t off = 0;
        if (m < n) {
            const int r = a.rows ? a.rows[m] : m;
            if (r < 0 || r >= a.h_rows) {
                if (rank == 0) record_fault(ws, TEE_DEVERR_ROW, r);
            } else {
                p = a.pos ? a.pos[r] : a.pos0 + r;
                const int s = a.seq ? a.seq[r] : 0;
                if (!pos_ok(p, a.cl.max_pos, a.hdr)) {
                    if (rank == 0) record_fault(ws, TEE_DEVERR_POS, p);
                } else if (s < 0 || s >= a.cl.n_seq) {
                    if (rank == 0) record_fault(ws, TEE_DEVERR_SEQ, s);
                } else {
                    good = 1;
                    off = L.cache_layer * a.cl.s_layer + s * a.cl.s_seq + static_cast<int64_t>(p) * a.cl.s_pos;
                }
            }
            // Rows are staged when in range, whatever the slot check says.
            ok[m] = (r >= 0 && r < a.h_rows) ? (good ? 2 : 1) : 0;
        } else {
            ok[m] = 0;
        }
        ps[m] = p;
        offs[m] = off;
    }
    __syncthreads();

    // 1. h rows -> As (fp32), eight elements per load; rows out of range read as zero.
    {
        const int per_row = d / 8;
        for (int i = threadIdx.x; i < n * per_row; i += SF_THREADS) {
            const int m = i / per_row, c = (i - m * per_row) * 8;
            float f[8];
            if (ok[m]) {
                const int r = a.rows ? a.rows[m] : m;
                load8(static_cast<const T*>(a.h) + static_cast<int64_t>(r) * a.ld_h + c, f);
            } else {
#pragma unroll
                for (int q = 0; q < 8; ++q) f[q] = 0.f;
            }
            reinterpret_cast<float4*>(As + m * d + c)[0] = make_float4(f[0], f[1], f[2], f[3]);
            reinterpret_cast<float4*>(As + m * d + c)[1] = make_float4(f[4], f[5], f[6], f[7]);
        }
    }
    if (a.stage) asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();

    // 2. x (map or identity), 1 / rms(x), x^ = x * rs * gamma in As.
    if (wmap) {
        for (int c = 0; c < cpc; c += 32) {
            if (a.stage)
                col_pass<T, NM>(As, d, n, d, reinterpret_cast<const T*>(w_map_s), cpc, c, min(32, cpc - c), red, xs,
                                cpc, c);
            else
                col_pass<T, NM>(As, d, n, d, wmap, d, rank * cpc + c, min(32, cpc - c), red, xs, cpc, c);
        }
        for (int m = warp; m < n; m += SF_WARPS) {
            float s = 0.f;
            for (int c = lane; c < cpc; c += 32) s = fmaf(xs[m * cpc + c], xs[m * cpc + c], s);
            s = warp_sum(s);
            if (lane == 0) ssp[m] = s;
        }
        sf_cluster_arrive();
        sf_cluster_wait();   // every CTA's slice and partial sums are complete
        if (threadIdx.x < n) {   // the eight partial sums: every load issued before the first add
            const int m = threadIdx.x;
            float v[SF_CLUSTER];
#pragma unroll
            for (int q = 0; q < SF_CLUSTER; ++q) v[q] = sf_ld_peer(ssp + m, q);
            float s = 0.f;
#pragma unroll
            for (int q = 0; q < SF_CLUSTER; ++q) s += v[q];
            rs[m] = 1.0f / sqrtf(s / static_cast<float>(d) + a.eps);
        }
        __syncthreads();
        // x^ rows from the eight slices: 16-byte loads, four per thread in flight
        const int c4n = cpc / 4, per_m = SF_CLUSTER * c4n, total4 = n * per_m;
        for (int i0 = threadIdx.x; i0 < total4; i0 += 4 * SF_THREADS) {
            float4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u * SF_THREADS;
                if (i < total4) {
                    const int m = i / per_m, r = i - m * per_m, q = r / c4n, c4 = r - q * c4n;
                    v[u] = sf_ld_peer4(xs + m * cpc + 4 * c4, q);
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u * SF_THREADS;
                if (i < total4) {
                    const int m = i / per_m, r = i - m * per_m, q = r / c4n, c4 = r - q * c4n;
                    const int k = q * cpc + 4 * c4;
                    const float sc = rs[m];
                    float* dst = As + m * d + k;
                    dst[0] = v[u].x * sc * to_f32(gamma[k]);
                    dst[1] = v[u].y * sc * to_f32(gamma[k + 1]);
                    dst[2] = v[u].z * sc * to_f32(gamma[k + 2]);
                    dst[3] = v[u].w * sc * to_f32(gamma[k + 3]);
                }
            }
        }
        sf_cluster_arrive();   // this CTA has read its peers' slices (waited on before exit)
    } else {
        for (int m = warp; m < n; m += SF_WARPS) {
            float s = 0.f;
            for (int k = lane; k < d; k += 32) s = fmaf(As[m * d + k], As[m * d + k], s);
            s = warp_sum(s);
            if (lane == 0) rs[m] = 1.0f / sqrtf(s / static_cast<float>(d) + a.eps);
        }
        __syncthreads();
        for (int i = threadIdx.x; i < n * d; i += SF_THREADS) {
            const int m = i / d, k = i - m * d;
            As[i] *= rs[m] * to_f32(gamma[k]);
        }
    }
    __syncthreads();

    // 3. this CTA's heads.
    const float2* rope = a.rope;
    int slot = 0;
    for (int hh = rank; hh < 2 * a.n_kv; hh += SF_CLUSTER, ++slot) {
        const bool is_k = hh < a.n_kv;
        if (is_k ? !write_k : !write_v) continue;
        const int h = is_k ? hh : hh - a.n_kv;
        const T* w = static_cast<const T*>(is_k ? L.wk : L.wv);
        const T* ws_h = reinterpret_cast<const T*>(w_head_s + static_cast<size_t>(slot) * d * hd * es);
        for (int c = 0; c < hd; c += 32) {
            if (a.stage)
                col_pass<T, NM>(As, d, n, d, ws_h, hd, c, min(32, hd - c), red, hv, hd, c);
            else
                col_pass<T, NM>(As, d, n, d, w, kvw, h * hd + c, min(32, hd - c), red, hv, hd, c);
        }
        const T* bias = static_cast<const T*>(is_k ? L.k_bias : L.v_bias);
        const T* kn = is_k ? static_cast<const T*>(L.k_norm) : nullptr;
        T* cache = static_cast<T*>(is_k ? a.k_cache : a.v_cache);
        for (int m = warp; m < n; m += SF_WARPS) {
            if (ok[m] != 2) continue;
            float* v = hv + m * hd;
            if (bias)
                for (int i = lane; i < hd; i += 32) v[i] += to_f32(bias[h * hd + i]);
            float krs = 1.f;
            if (kn) {
                __syncwarp();
                float s = 0.f;
                for (int i = lane; i < hd; i += 32) s = fmaf(v[i], v[i], s);
                krs = 1.0f / sqrtf(warp_sum(s) / static_cast<float>(hd) + a.eps);
            }
            __syncwarp();
            T* dst = cache + offs[m] + h * a.cl.s_head;
            const int p = ps[m];
            for (int i = lane; i < half; i += 32) {
                float x1 = v[i], x2 = v[i + half];
                if (is_k) {
                    if (kn) {
                        x1 *= krs * to_f32(kn[i]);
                        x2 *= krs * to_f32(kn[i + half]);
                    }
                    const float2 cs = rope[static_cast<int64_t>(p) * half + i];
                    const float y1 = x1 * cs.x - x2 * cs.y, y2 = x2 * cs.x + x1 * cs.y;
                    x1 = y1;
                    x2 = y2;
                }
                dst[i] = from_f32<T>(x1);
                dst[i + half] = from_f32<T>(x2);
            }
        }
        __syncthreads();   // hv is rewritten by the next head
    }
    if (wmap) sf_cluster_wait();   // peers are done reading this CTA's slice
}

constexpr size_t SF_SMEM_MAX = 220 * 1024;

template <typename T, int NM>
tee_status launch_small(SmallArgs a, int n_layers, bool stage_ok, void* ws, cudaStream_t s) {
    const SmallLayout lay = small_layout(a.n_max, a.d, a.hd, NM, a.n_kv, sizeof(T), a.has_map);
    a.stage = stage_ok && lay.staged_bytes <= SF_SMEM_MAX;
    const size_t smem = a.stage ? lay.staged_bytes : lay.bytes;
    static bool attr_set = false;
    if (!attr_set) {
        tee_status st = cuda_status(cudaFuncSetAttribute(fill_small_kernel<T, NM>,
                                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                         static_cast<int>(SF_SMEM_MAX)));
        if (st != TEE_OK) return st;
        attr_set = true;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(SF_CLUSTER, n_layers);
    cfg.blockDim = dim3(SF_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.early ? 1 : 0;
    const tee_status st = cuda_status(cudaLaunchKernelEx(&cfg, fill_small_kernel<T, NM>, a, ws));
    return st != TEE_OK ? st : launch_status();
}

template <typename T>
tee_status run_small(const FillCall& fc) {
    const tee_fill_desc& D = *fc.desc;
    const PrepView pv = prep_view(fc.prep, D, fc.n_layers);
    SmallArgs a{};
    a.n_max = fc.n_max;
    a.n_dev = fc.n_dev;
    a.d = D.d;
    a.n_kv = D.n_kv_heads;
    a.hd = D.head_dim;
    a.eps = D.eps;
    a.h = fc.h;
    a.ld_h = fc.ld_h;
    a.h_rows = fc.h_rows;
    a.rows = fc.rows;
    a.pos = fc.pos;
    a.pos0 = fc.pos0;
    a.seq = fc.seq;
    a.hdr = pv.hdr;
    a.rope = pv.rope;
    a.k_cache = fc.k_cache;
    a.v_cache = fc.v_cache;
    a.cl = *fc.cache;
    // Staging copies 16-byte pieces: rows of the map slice and of a head must be
    // whole pieces, and the weights 16-byte aligned.
    const size_t es = sizeof(T);
    for (int l0 = 0; l0 < fc.n_layers; l0 += SF_MAX_LAYERS) {
        const int nl = fc.n_layers - l0 < SF_MAX_LAYERS ? fc.n_layers - l0 : SF_MAX_LAYERS;
        bool stage_ok = (D.head_dim * es) % 16 == 0;
        a.has_map = 0;
        for (int i = 0; i < nl; ++i) {
            const tee_fill_layer& L = fc.layers[l0 + i];
            a.l[i] = SmallLayer{L.w_map, L.gamma, L.wk, L.wv, L.k_bias, L.v_bias, L.k_norm, L.cache_layer, L.writes};
            if (L.w_map) {
                a.has_map = 1;
                stage_ok = stage_ok && aligned16(L.w_map) && ((D.d / SF_CLUSTER) * es) % 16 == 0;
            }
            stage_ok = stage_ok && aligned16(L.wk) && aligned16(L.wv);
        }
        // Only the first launch may overlap the kernel before the call.
        a.early = (l0 == 0 && (D.flags & TEE_FILL_EARLY_WEIGHTS)) ? 1 : 0;
        const tee_status st = fc.n_max <= 8 ? launch_small<T, 8>(a, nl, stage_ok, fc.ws, fc.stream)
                                            : launch_small<T, SF_MAX_ITEMS>(a, nl, stage_ok, fc.ws, fc.stream);
        if (st != TEE_OK) return st;
    }
    return TEE_OK;
}

}  // namespace

tee_status fill_small_run(const FillCall& fc) {
    const tee_fill_desc& D = *fc.desc;
    if (D.wfmt != TEE_W_DENSE || fc.n_max > SF_MAX_ITEMS || D.d % 32 || D.d > SF_MAX_D ||
        static_cast<int64_t>(fc.n_max) * D.d > SF_MAX_ELEMS || D.head_dim > SF_MAX_HD || D.head_dim % 2)
        return TEE_ERR_UNSUPPORTED;
    switch (D.dtype) {
        case TEE_F32: return run_small<float>(fc);
        case TEE_F16: return run_small<__half>(fc);
        default: return run_small<__nv_bfloat16>(fc);
    }
}

}  // namespace tee
