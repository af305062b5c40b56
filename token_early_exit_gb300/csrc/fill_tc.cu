// Tensor-core (tcgen05) path of the KV fill for large bf16 fills with dense
// weights (RidgeFill prefill: thousands to ~10^5 rows per call).
//
// Per filled layer j, two persistent GEMMs on the 5th-generation tensor cores:
//   GEMM1 (map)  X = h_split . W_j            epilogue: store X as bf16 and
//                                             accumulate sum(X^2) per row
//   GEMM2 (K/V)  [K|V] = X . (diag(g_j)[Wk_j|Wv_j])
//                                             epilogue: scale by 1/rms(X),
//                                             RoPE on K, store to the cache
// RMSNorm is diag(1/rms(x)) x diag(g): the row scale commutes out of the
// projection, so g_j is folded into the K-major projection weights once in
// prepare, and 1/rms is applied in GEMM2's epilogue. With an identity map
// GEMM1 is skipped and a row-norm kernel provides sum(h^2).
//
// GEMM structure (one CTA per SM, persistent over 128 x 256 output tiles):
// warp 4 issues TMA loads of 128x64 A and 256x64 B bf16 tiles (128-byte
// swizzle) into a 4-stage shared-memory ring; one thread of warp 5 issues
// tcgen05.mma (M=128, N=256, K=16) into one of two TMEM accumulators
// (2 x 256 fp32 columns) and commits to the ring's "empty" barriers; warps
// 0-3 read the finished accumulator with tcgen05.ld (one row per thread) and
// run the epilogue while the next tile accumulates in the other buffer.
#include <cudaTypedefs.h>

#include <mutex>

#include "fill.cuh"
#include "tc.cuh"

namespace tee {

// ------------------------------------------------------------------ tensor maps
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static std::once_flag g_encode_once;

static bool encoder_ready() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

tee_status make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t row_bytes,
                          uint32_t box_inner, uint32_t box_rows) {
    if (!encoder_ready()) return TEE_ERR_UNSUPPORTED;
    if (inner == 0 || rows == 0) return TEE_ERR_INVALID_ARG;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? TEE_OK : TEE_ERR_INVALID_ARG;
}

tee_status make_tmap_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t row_bytes,
                        uint32_t box_inner, uint32_t box_rows) {
    if (!encoder_ready()) return TEE_ERR_UNSUPPORTED;
    if (inner == 0 || rows == 0) return TEE_ERR_INVALID_ARG;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? TEE_OK : TEE_ERR_INVALID_ARG;
}

tee_status make_tmap_cache(CUtensorMap* map, const void* base, int head_dim, const tee_cache_layout& cl,
                           uint32_t box_rows) {
    if (!encoder_ready()) return TEE_ERR_UNSUPPORTED;
    cuuint64_t dims[5] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(cl.max_pos),
                          static_cast<cuuint64_t>(cl.n_heads), static_cast<cuuint64_t>(cl.n_seq),
                          static_cast<cuuint64_t>(cl.n_layers)};
    cuuint64_t strides[4] = {static_cast<cuuint64_t>(cl.s_pos) * 2, static_cast<cuuint64_t>(cl.s_head) * 2,
                             static_cast<cuuint64_t>(cl.s_seq) * 2, static_cast<cuuint64_t>(cl.s_layer) * 2};
    cuuint32_t box[5] = {64, box_rows, 1, 1, 1};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? TEE_OK : TEE_ERR_INVALID_ARG;
}

// A K-major bf16 matrix [rows][n_kb * 64] seen as n_kb blocks of 64 columns: one
// box brings box_kb consecutive blocks of box_rows rows, each block landing as its
// own 128-byte-swizzled [box_rows][64] tile (block stride 128 bytes in the source).
tee_status make_tmap_bf16_kblocks(CUtensorMap* map, const void* base, uint64_t rows, uint64_t row_bytes,
                                  uint64_t n_kb, uint32_t box_rows, uint32_t box_kb) {
    if (!encoder_ready()) return TEE_ERR_UNSUPPORTED;
    if (rows == 0 || n_kb == 0) return TEE_ERR_INVALID_ARG;
    cuuint64_t dims[3] = {64, rows, n_kb};
    cuuint64_t strides[2] = {row_bytes, 128};
    cuuint32_t box[3] = {64, box_rows, box_kb};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? TEE_OK : TEE_ERR_INVALID_ARG;
}

namespace {

using bf16 = __nv_bfloat16;

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4, EPI_WARPS = 4;
constexpr int THREADS = (EPI_WARPS + 2) * 32;
constexpr uint32_t A_BYTES = BM * BK * 2, B_BYTES = BN * BK * 2, STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr size_t SMEM_BYTES = 1024 + size_t(STAGES) * STAGE_BYTES + 256;

enum { EPI_MAP = 0, EPI_KV = 1, EPI_F32 = 2 };
// Where a pipeline wait gave up (detail of TEE_DEVERR_TIMEOUT).
enum { W_EMPTY = 1, W_ACC_EMPTY = 2, W_FULL = 3, W_ACC_FULL = 4, W_DRAIN = 5, W_TEARDOWN = 6 };

struct EpiArgs {
    // GEMM1: X and its row sums of squares
    bf16* x;
    int64_t ldx;
    float* sumsq_out;
    // GEMM2: the cache store
    const float* sumsq_in;
    float inv_d, eps;
    const int32_t* pos;
    int pos0;
    const int32_t* seq;
    const PrepHeader* hdr;
    const float2* rope;
    bf16* kc;
    bf16* vc;
    tee_cache_layout cl;
    int layer, kvw, hd, half, h_rows;
    // the GEMM's column 0 is output column col_off of [K|V] (kvw for a V-only layer);
    // per-layer bias of K and V and per-head K norm weight (all nullable)
    int col_off;
    const bf16* kb;
    const bf16* vb;
    const bf16* kn;
    // fp32 output (the ridge fit's Gram matrices): C, its row stride, and a value
    // added where row == column; with sub the product is subtracted from C instead
    // (the ridge fit's substitution updates)
    float* c32;
    int64_t ldc32;
    float diag;
    int sub;
};

__device__ __forceinline__ void store32_bf16(bf16* dst, const float (&v)[32]) {
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q)
        d[q] = make_uint4(pack_bf16x2(v[8 * q + 0], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                          pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
}

// Map epilogue: X tile row -> bf16 store, sum of squares of the fp32 values.
__device__ __forceinline__ void epi_map(const EpiArgs& ep, int row, int n, int c0, uint32_t t_base) {
    const bool ok = row < n;
    float ss = 0.f;
    bf16* dst = ep.x + static_cast<int64_t>(row) * ep.ldx + c0;
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
        float v[32];
        tc::tmem_ld32(t_base + c * 32, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) ss = fmaf(v[j], v[j], ss);
        if (ok) store32_bf16(dst + c * 32, v);
    }
    if (ok) atomicAdd(ep.sumsq_out + row, ss);
}

// fp32 epilogue: the tile row as it accumulated, plus ep.diag on the diagonal.
__device__ __forceinline__ void epi_f32(const EpiArgs& ep, int row, int n, int c0, uint32_t t_base) {
    const bool ok = row < n;
    float* dst = ep.c32 + static_cast<int64_t>(row) * ep.ldc32 + c0;
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
        float v[32];
        tc::tmem_ld32(t_base + c * 32, v);
        if (!ok) continue;
        float4* d4 = reinterpret_cast<float4*>(dst + c * 32);
        if (ep.sub) {
            float4 o[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) o[q] = d4[q];
#pragma unroll
            for (int q = 0; q < 8; ++q)
                d4[q] = make_float4(o[q].x - v[4 * q], o[q].y - v[4 * q + 1], o[q].z - v[4 * q + 2], o[q].w - v[4 * q + 3]);
            continue;
        }
        const int dc = row - (c0 + c * 32);
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (j == dc) v[j] += ep.diag;
#pragma unroll
        for (int q = 0; q < 8; ++q) d4[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    }
}

__device__ __forceinline__ void load32_bf16(const bf16* src, float (&v)[32]) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint4 u = s4[q];
        unpack_bf16x2(u.x, v[8 * q + 0], v[8 * q + 1]);
        unpack_bf16x2(u.y, v[8 * q + 2], v[8 * q + 3]);
        unpack_bf16x2(u.z, v[8 * q + 4], v[8 * q + 5]);
        unpack_bf16x2(u.w, v[8 * q + 6], v[8 * q + 7]);
    }
}

// K/V epilogue: 1/rms row scale, bias, the per-head K norm, RoPE on K heads,
// store into the cache slot.
__device__ __forceinline__ void epi_kv(const EpiArgs& ep, int row, int n, int c0, uint32_t t_base, void* ws) {
    bool ok = row < n;
    float r = 0.f;
    int p = 0, s = 0;
    if (ok) {
        if (row >= ep.h_rows) {
            if (c0 == 0) record_fault(ws, TEE_DEVERR_ROW, row);
            ok = false;
        } else {
            r = 1.0f / sqrtf(ep.sumsq_in[row] * ep.inv_d + ep.eps);
            p = ep.pos ? ep.pos[row] : ep.pos0 + row;
            s = ep.seq ? ep.seq[row] : 0;
            if (!pos_ok(p, ep.cl.max_pos, ep.hdr)) {
                if (c0 == 0) record_fault(ws, TEE_DEVERR_POS, p);
                ok = false;
            } else if (s < 0 || s >= ep.cl.n_seq) {
                if (c0 == 0) record_fault(ws, TEE_DEVERR_SEQ, s);
                ok = false;
            }
        }
    }
    const int cg = c0 + ep.col_off;
    const bool is_k = cg < ep.kvw;
    const int col0 = is_k ? cg : cg - ep.kvw;
    bf16* cache = is_k ? ep.kc : ep.vc;
    const bf16* bias = is_k ? ep.kb : ep.vb;
    const bool knorm = is_k && ep.kn;
    const int64_t base = ep.layer * ep.cl.s_layer + s * ep.cl.s_seq + static_cast<int64_t>(p) * ep.cl.s_pos;
    const float2* cs = ep.rope + static_cast<int64_t>(p) * ep.half;
#pragma unroll 1
    for (int hb = 0; hb < BN; hb += ep.hd) {
        bf16* dst = cache + base + static_cast<int64_t>((col0 + hb) / ep.hd) * ep.cl.s_head;
        const bf16* bh = bias ? bias + col0 + hb : nullptr;
        // QK-norm: a first pass over the head for the RMS of r * acc + bias
        float hs = 1.f;
        if (knorm) {
            float ss = 0.f;
#pragma unroll 1
            for (int c = 0; c < ep.hd; c += 32) {
                float v[32], b[32];
                tc::tmem_ld32(t_base + hb + c, v);
                if (bh) load32_bf16(bh + c, b);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float a = bh ? fmaf(v[j], r, b[j]) : v[j] * r;
                    ss = fmaf(a, a, ss);
                }
            }
            hs = 1.0f / sqrtf(ss / static_cast<float>(ep.hd) + ep.eps);
        }
#pragma unroll 1
        for (int c = 0; c < ep.half; c += 32) {
            float lo[32], hi[32];
            tc::tmem_ld32(t_base + hb + c, lo);
            tc::tmem_ld32(t_base + hb + ep.half + c, hi);
            if (!ok) continue;
            if (bh) {
                float b[32];
                load32_bf16(bh + c, b);
#pragma unroll
                for (int j = 0; j < 32; ++j) lo[j] = fmaf(lo[j], r, b[j]);
                load32_bf16(bh + ep.half + c, b);
#pragma unroll
                for (int j = 0; j < 32; ++j) hi[j] = fmaf(hi[j], r, b[j]);
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    lo[j] *= r;
                    hi[j] *= r;
                }
            }
            if (knorm) {
                float g[32];
                load32_bf16(ep.kn + c, g);
#pragma unroll
                for (int j = 0; j < 32; ++j) lo[j] *= hs * g[j];
                load32_bf16(ep.kn + ep.half + c, g);
#pragma unroll
                for (int j = 0; j < 32; ++j) hi[j] *= hs * g[j];
            }
            if (is_k) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float2 e = cs[c + j];
                    const float a = lo[j], b = hi[j];
                    lo[j] = a * e.x - b * e.y;
                    hi[j] = b * e.x + a * e.y;
                }
            }
            store32_bf16(dst + c, lo);
            store32_bf16(dst + ep.half + c, hi);
        }
    }
}

template <int EPI>
__global__ void __launch_bounds__(THREADS, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, int n_max,
               const int32_t* __restrict__ n_dev, int N, int K, EpiArgs ep, void* ws) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* acc_full = empty + STAGES;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* drain = acc_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = item_count(n_max, n_dev);
    const int n_tiles = N / BN, k_blocks = K / BK;
    const int total = ((n + BM - 1) / BM) * n_tiles;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&acc_full[b], 1);
            tc::mbar_init(&acc_empty[b], EPI_WARPS);
        }
        tc::mbar_init(drain, 1);
        *abort = 0;
        tc::fence_barrier_init();
    }
    if (warp == EPI_WARPS + 1) tc::tmem_alloc(tmem_slot, TMEM_COLS);
    if (warp == EPI_WARPS && lane == 0) {
        tc::prefetch_tmap(&tmA);
        tc::prefetch_tmap(&tmB);
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == EPI_WARPS) {
        // ---------------- TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, issued_phase = 0;  // per-stage bits: loads issued / parity of the last issue
            bool stop = false;
            for (int t = blockIdx.x; t < total && !stop; t += gridDim.x) {
                const int m0 = (t / n_tiles) * BM, c0 = (t % n_tiles) * BN;
                for (int kb = 0; kb < k_blocks; ++kb) {
                    if (!tc::mbar_wait(&empty[stage], phase ^ 1, abort, ws, W_EMPTY)) {
                        stop = true;
                        break;
                    }
                    uint8_t* sa = smem + stage * STAGE_BYTES;
                    tc::mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
                    tc::tma_load_2d(sa, &tmA, kb * BK, m0, &full[stage]);
                    tc::tma_load_2d(sa + A_BYTES, &tmB, kb * BK, c0, &full[stage]);
                    issued |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (*abort) {
                // Let copies still in flight land before the block's shared memory goes away.
                for (int s = 0; s < STAGES; ++s) {
                    if (!(issued >> s & 1)) continue;
                    const uint32_t par = issued_phase >> s & 1;
                    const uint64_t t0 = tc::globaltimer();
                    while (!tc::mbar_try_wait(&full[s], par) && tc::globaltimer() - t0 < tc::WAIT_LIMIT_NS) {
                    }
                }
            }
        }
    } else if (warp == EPI_WARPS + 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            constexpr uint32_t idesc = tc::idesc_bf16(BM, BN);
            bool stop = false;
            for (int t = blockIdx.x; t < total && !stop; t += gridDim.x) {
                if (!tc::mbar_wait(&acc_empty[acc], acc_phase ^ 1, abort, ws, W_ACC_EMPTY)) break;
                tc::tc_fence_after();
                const uint32_t d_tmem = tmem + acc * BN;
                for (int kb = 0; kb < k_blocks; ++kb) {
                    if (!tc::mbar_wait(&full[stage], phase, abort, ws, W_FULL)) {
                        stop = true;
                        break;
                    }
                    tc::tc_fence_after();
                    const uint32_t sa = tc::smem_u32(smem + stage * STAGE_BYTES);
                    const uint64_t ad = tc::smem_desc_sw128(sa), bd = tc::smem_desc_sw128(sa + A_BYTES);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        tc::umma_bf16(d_tmem, ad + 2 * k, bd + 2 * k, idesc, (kb | k) != 0);
                    tc::umma_commit(&empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (stop) break;
                tc::umma_commit(&acc_full[acc]);
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1;
                }
            }
            // Every MMA issued above has finished once the drain barrier flips.
            tc::umma_commit(drain);
            const uint64_t t0 = tc::globaltimer();
            while (!tc::mbar_try_wait(drain, 0)) {
                if (tc::globaltimer() - t0 > tc::WAIT_LIMIT_NS) {
                    *abort = 1;
                    record_fault(ws, TEE_DEVERR_TIMEOUT, W_DRAIN);
                    break;
                }
            }
        }
    } else {
        // ---------------- epilogue warps 0..3 (TMEM lane quadrant = warp)
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x) {
            if (!tc::mbar_wait(&acc_full[acc], acc_phase, abort, ws, W_ACC_FULL)) break;
            tc::tc_fence_after();
            const int m0 = (t / n_tiles) * BM, c0 = (t % n_tiles) * BN;
            const int row = m0 + warp * 32 + lane;
            const uint32_t t_base = tmem + (static_cast<uint32_t>(warp * 32) << 16) + acc * BN;
            if (EPI == EPI_MAP)
                epi_map(ep, row, n, c0, t_base);
            else if (EPI == EPI_KV)
                epi_kv(ep, row, n, c0, t_base, ws);
            else
                epi_f32(ep, row, n, c0, t_base);
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&acc_empty[acc]);
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1;
            }
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == EPI_WARPS + 1) tc::tmem_dealloc(tmem, TMEM_COLS);
}

// sumsq[i] = sum_k h[i][k]^2 for the identity map (x_j = h).
__global__ void __launch_bounds__(256)
row_sumsq_kernel(int n_max, const int32_t* __restrict__ n_dev, int h_rows, int d, const bf16* __restrict__ h,
                 int64_t ldh, float* __restrict__ sumsq) {
    const int n = min(item_count(n_max, n_dev), h_rows);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int m = blockIdx.x * 8 + warp; m < n; m += gridDim.x * 8) {
        const bf16* x = h + static_cast<int64_t>(m) * ldh;
        float ss = 0.f;
        for (int k = lane * 8; k < d; k += 256) {
            float v[8];
            load8(x + k, v);
#pragma unroll
            for (int q = 0; q < 8; ++q) ss = fmaf(v[q], v[q], ss);
        }
        ss = warp_sum(ss);
        if (lane == 0) sumsq[m] = ss;
    }
}

// out[c][k] = in[k][c] * g[k] (g nullable): K-major copy of a [K][C] matrix.
__global__ void transpose_scale_kernel(const bf16* __restrict__ in, int K, int C, int64_t ld_in,
                                       const bf16* __restrict__ g, bf16* __restrict__ out, int64_t ld_out) {
    __shared__ float tile[32][33];
    const int k0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int k = k0 + i, c = c0 + threadIdx.x;
        float v = 0.f;
        if (k < K && c < C) {
            v = __bfloat162float(in[static_cast<int64_t>(k) * ld_in + c]);
            if (g) v *= __bfloat162float(g[k]);
        }
        tile[i][threadIdx.x] = v;
    }
    __syncthreads();
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int c = c0 + i, k = k0 + threadIdx.x;
        if (c < C && k < K) out[static_cast<int64_t>(c) * ld_out + k] = __float2bfloat16_rn(tile[threadIdx.x][i]);
    }
}

bool desc_eligible(const tee_fill_desc& D) {
    const int kvw = D.n_kv_heads * D.head_dim;
    return D.dtype == TEE_BF16 && D.wfmt == TEE_W_DENSE && D.d % BK == 0 && D.d % BN == 0 &&
           (D.head_dim == 64 || D.head_dim == 128 || D.head_dim == 256) && kvw % BN == 0;
}

size_t layer_bytes(const tee_fill_desc& D) {
    const size_t d = D.d, kvw = static_cast<size_t>(D.n_kv_heads) * D.head_dim;
    return round_up(d * d * 2, 1024) + round_up(2 * kvw * d * 2, 1024);
}

struct TcWs {
    size_t sumsq_off, x_off, end;
};
TcWs tc_ws(const tee_fill_desc& D, int n_layers, int n_max) {
    TcWs w;
    w.sumsq_off = TEE_WS_HEADER_BYTES;
    w.x_off = round_up(w.sumsq_off + static_cast<size_t>(n_layers) * n_max * 4, 1024);
    w.end = round_up(w.x_off + static_cast<size_t>(n_max) * D.d * 2, 1024);
    return w;
}

template <int EPI>
tee_status launch_gemm(const CUtensorMap& a, const CUtensorMap& b, int n_max, const int32_t* n_dev, int N, int K,
                       const EpiArgs& ep, void* ws, cudaStream_t s) {
    static bool attr_set = false;
    if (!attr_set) {
        tee_status st = cuda_status(cudaFuncSetAttribute(tc_gemm_kernel<EPI>,
                                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                         static_cast<int>(SMEM_BYTES)));
        if (st != TEE_OK) return st;
        attr_set = true;
    }
    const int tiles = ((n_max + BM - 1) / BM) * (N / BN);
    int grid = sm_count();
    if (grid > tiles) grid = tiles;
    if (grid < 1) grid = 1;
    tc_gemm_kernel<EPI><<<grid, THREADS, SMEM_BYTES, s>>>(a, b, n_max, n_dev, N, K, ep, ws);
    return launch_status();
}

}  // namespace

// ---- the ridge fit's Gram matrices (RidgeFill's closed-form fit) on the same GEMM:
// G = X^T X + lambda I [d][d] and R = X^T Y [d][d_out], fp32, from bf16 X [n][ld_x]
// and Y [n][ld_y]. X and Y are first transposed into K-major copies [d][n_pad] and
// [d_out][n_pad] (n_pad = n rounded up to 64, zero columns past n).
size_t ridge_gram_ws_bytes(int n, int d, int d_out) {
    const size_t n_pad = round_up(static_cast<size_t>(n), BK);
    return round_up(static_cast<size_t>(d) * n_pad * 2, 1024) + round_up(static_cast<size_t>(d_out) * n_pad * 2, 1024);
}

tee_status ridge_gram(int n, int d, int d_out, const void* x, int64_t ld_x, const void* y, int64_t ld_y, float lambda,
                      float* g, float* r, int64_t ld_r, char* scratch, void* ws, cudaStream_t s) {
    if (d % BN || d_out % BN) return TEE_ERR_UNSUPPORTED;
    const int n_pad = static_cast<int>(round_up(static_cast<size_t>(n), BK));
    bf16* xt = reinterpret_cast<bf16*>(scratch);
    bf16* yt = reinterpret_cast<bf16*>(scratch + round_up(static_cast<size_t>(d) * n_pad * 2, 1024));
    tee_status st = cuda_status(cudaMemsetAsync(scratch, 0, ridge_gram_ws_bytes(n, d, d_out), s));
    if (st != TEE_OK) return st;
    dim3 blk(32, 8);
    transpose_scale_kernel<<<dim3((d + 31) / 32, (n + 31) / 32), blk, 0, s>>>(static_cast<const bf16*>(x), n, d, ld_x,
                                                                            nullptr, xt, n_pad);
    if ((st = launch_status()) != TEE_OK) return st;
    transpose_scale_kernel<<<dim3((d_out + 31) / 32, (n + 31) / 32), blk, 0, s>>>(static_cast<const bf16*>(y), n, d_out,
                                                                                ld_y, nullptr, yt, n_pad);
    if ((st = launch_status()) != TEE_OK) return st;
    CUtensorMap tx, ty;
    if ((st = make_tmap_bf16(&tx, xt, n_pad, d, static_cast<uint64_t>(n_pad) * 2, BK, BM)) != TEE_OK) return st;
    CUtensorMap txb;
    if ((st = make_tmap_bf16(&txb, xt, n_pad, d, static_cast<uint64_t>(n_pad) * 2, BK, BN)) != TEE_OK) return st;
    if ((st = make_tmap_bf16(&ty, yt, n_pad, d_out, static_cast<uint64_t>(n_pad) * 2, BK, BN)) != TEE_OK) return st;
    EpiArgs ep{};
    ep.c32 = g;
    ep.ldc32 = d;
    ep.diag = lambda;
    if ((st = launch_gemm<EPI_F32>(tx, txb, d, nullptr, d, n_pad, ep, ws, s)) != TEE_OK) return st;
    ep.c32 = r;
    ep.ldc32 = ld_r;
    ep.diag = 0.f;
    return launch_gemm<EPI_F32>(tx, ty, d, nullptr, d_out, n_pad, ep, ws, s);
}

// ---- the ridge fit's substitution updates on the same GEMM: C [M][N] (row stride
// ldc, fp32) -= A B^T with A [M][k3] and B [N][k3] bf16 (K-major rows, k3 a multiple
// of 64): the fp32 factors split into bf16 high and low parts, laid along K so that
// the one product carries a_hi b_hi + a_lo b_hi + a_hi b_lo.
tee_status ridge_update_tc(int M, int N, int k3, const void* a3, const void* b3, float* c, int64_t ldc, void* ws,
                           cudaStream_t s) {
    if (M <= 0) return TEE_OK;
    if (N % BN || k3 % BK) return TEE_ERR_UNSUPPORTED;
    CUtensorMap ta, tb;
    tee_status st = make_tmap_bf16(&ta, a3, k3, M, static_cast<uint64_t>(k3) * 2, BK, BM);
    if (st != TEE_OK) return st;
    if ((st = make_tmap_bf16(&tb, b3, k3, N, static_cast<uint64_t>(k3) * 2, BK, BN)) != TEE_OK) return st;
    EpiArgs ep{};
    ep.c32 = c;
    ep.ldc32 = ldc;
    ep.sub = 1;
    return launch_gemm<EPI_F32>(ta, tb, M, nullptr, N, k3, ep, ws, s);
}

size_t fill_tc_prep_bytes(const tee_fill_desc& D, int n_layers) {
    if (!desc_eligible(D)) return 0;
    return static_cast<size_t>(n_layers) * layer_bytes(D);
}

tee_status fill_tc_prepare(const tee_fill_desc& D, int n_layers, const tee_fill_layer* layers, char* tc_area,
                           cudaStream_t s) {
    if (!desc_eligible(D)) return TEE_OK;
    const int d = D.d, kvw = D.n_kv_heads * D.head_dim;
    for (int l = 0; l < n_layers; ++l) {
        const tee_fill_layer& L = layers[l];
        if (!L.gamma || !L.wk || !L.wv) return TEE_ERR_INVALID_ARG;
        bf16* wmap_t = reinterpret_cast<bf16*>(tc_area + l * layer_bytes(D));
        bf16* wkv_t = reinterpret_cast<bf16*>(reinterpret_cast<char*>(wmap_t) + round_up(size_t(d) * d * 2, 1024));
        dim3 blk(32, 8);
        if (L.w_map) {
            transpose_scale_kernel<<<dim3((d + 31) / 32, (d + 31) / 32), blk, 0, s>>>(
                static_cast<const bf16*>(L.w_map), d, d, d, nullptr, wmap_t, d);
            tee_status st = launch_status();
            if (st != TEE_OK) return st;
        }
        const bf16* g = static_cast<const bf16*>(L.gamma);
        transpose_scale_kernel<<<dim3((kvw + 31) / 32, (d + 31) / 32), blk, 0, s>>>(static_cast<const bf16*>(L.wk),
                                                                                     d, kvw, kvw, g, wkv_t, d);
        tee_status st = launch_status();
        if (st != TEE_OK) return st;
        transpose_scale_kernel<<<dim3((kvw + 31) / 32, (d + 31) / 32), blk, 0, s>>>(
            static_cast<const bf16*>(L.wv), d, kvw, kvw, g, wkv_t + static_cast<size_t>(kvw) * d, d);
        st = launch_status();
        if (st != TEE_OK) return st;
    }
    return TEE_OK;
}

size_t fill_tc_ws_bytes(const tee_fill_desc& D, int n_layers, int n_max) {
    if (!desc_eligible(D)) return 0;
    return tc_ws(D, n_layers, n_max).end;
}

// Smallest fill that goes to the tensor cores (fewer rows take the decode path).
constexpr int TC_MIN_ROWS = 256;

tee_status fill_tc_run(const FillCall& fc) {
    const tee_fill_desc& D = *fc.desc;
    if (!desc_eligible(D) || fc.rows || fc.n_max < TC_MIN_ROWS) return TEE_ERR_UNSUPPORTED;
    const tee_cache_layout& cl = *fc.cache;
    // 16-byte vector stores into the cache and 16-byte TMA rows.
    if (!aligned16(fc.k_cache) || !aligned16(fc.v_cache) || cl.s_layer % 8 || cl.s_seq % 8 || cl.s_head % 8 ||
        cl.s_pos % 8 || (fc.ld_h * 2) % 16)
        return TEE_ERR_UNSUPPORTED;
    const int d = D.d, kvw = D.n_kv_heads * D.head_dim, n_max = fc.n_max;
    const TcWs w = tc_ws(D, fc.n_layers, n_max);
    float* sumsq_all = ws_at<float>(fc.ws, w.sumsq_off);
    bf16* X = ws_at<bf16>(fc.ws, w.x_off);
    const PrepView pv = prep_view(fc.prep, D, fc.n_layers);
    tee_status st = cuda_status(
        cudaMemsetAsync(sumsq_all, 0, static_cast<size_t>(fc.n_layers) * n_max * 4, fc.stream));
    if (st != TEE_OK) return st;

    CUtensorMap tm_h, tm_x, tm_b;
    const uint64_t h_rows = static_cast<uint64_t>(fc.h_rows < n_max ? fc.h_rows : n_max);
    if (h_rows == 0) return TEE_OK;
    st = make_tmap_bf16(&tm_h, fc.h, d, h_rows, static_cast<uint64_t>(fc.ld_h) * 2, BK, BM);
    if (st != TEE_OK) return st;
    st = make_tmap_bf16(&tm_x, X, d, n_max, static_cast<uint64_t>(d) * 2, BK, BM);
    if (st != TEE_OK) return st;

    EpiArgs ep{};
    ep.x = X;
    ep.ldx = d;
    ep.inv_d = 1.0f / static_cast<float>(d);
    ep.eps = D.eps;
    ep.pos = fc.pos;
    ep.pos0 = fc.pos0;
    ep.seq = fc.seq;
    ep.hdr = pv.hdr;
    ep.rope = pv.rope;
    ep.kc = static_cast<bf16*>(fc.k_cache);
    ep.vc = static_cast<bf16*>(fc.v_cache);
    ep.cl = cl;
    ep.kvw = kvw;
    ep.hd = D.head_dim;
    ep.half = D.head_dim / 2;
    ep.h_rows = fc.h_rows;

    for (int l = 0; l < fc.n_layers; ++l) {
        const tee_fill_layer& L = fc.layers[l];
        const char* lb = pv.tc + l * layer_bytes(D);
        const bf16* wmap_t = reinterpret_cast<const bf16*>(lb);
        const bf16* wkv_t = reinterpret_cast<const bf16*>(lb + round_up(size_t(d) * d * 2, 1024));
        float* sumsq = sumsq_all + static_cast<size_t>(l) * n_max;
        const CUtensorMap* a2 = &tm_h;
        if (L.w_map) {
            st = make_tmap_bf16(&tm_b, wmap_t, d, d, static_cast<uint64_t>(d) * 2, BK, BN);
            if (st != TEE_OK) return st;
            ep.sumsq_out = sumsq;
            st = launch_gemm<EPI_MAP>(tm_h, tm_b, n_max, fc.n_dev, d, d, ep, fc.ws, fc.stream);
            if (st != TEE_OK) return st;
            a2 = &tm_x;
        } else {
            int blocks = (n_max + 7) / 8;
            if (blocks > 4096) blocks = 4096;
            row_sumsq_kernel<<<blocks, 256, 0, fc.stream>>>(n_max, fc.n_dev, fc.h_rows, d,
                                                           static_cast<const bf16*>(fc.h), fc.ld_h, sumsq);
            st = launch_status();
            if (st != TEE_OK) return st;
        }
        // a K-only or V-only layer multiplies by its half of [Wk|Wv] alone
        const int n_cols = L.writes ? kvw : 2 * kvw;
        ep.col_off = L.writes == TEE_FILL_WRITE_V ? kvw : 0;
        st = make_tmap_bf16(&tm_b, wkv_t + static_cast<size_t>(ep.col_off) * d, d, n_cols,
                            static_cast<uint64_t>(d) * 2, BK, BN);
        if (st != TEE_OK) return st;
        ep.sumsq_in = sumsq;
        ep.layer = L.cache_layer;
        ep.kb = static_cast<const bf16*>(L.k_bias);
        ep.vb = static_cast<const bf16*>(L.v_bias);
        ep.kn = static_cast<const bf16*>(L.k_norm);
        st = launch_gemm<EPI_KV>(*a2, tm_b, n_max, fc.n_dev, n_cols, d, ep, fc.ws, fc.stream);
        if (st != TEE_OK) return st;
    }
    return TEE_OK;
}

}  // namespace tee
