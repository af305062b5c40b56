// RidgeFill's per-layer linear map, fitted on the GPU (RidgeFill, "closed-form
// ridge regression" note): W = (X^T X + lambda I)^-1 X^T Y, with X the split-layer
// states and Y the true inputs of the filled layer over the calibration rows.
//
// The Gram matrices G = X^T X + lambda I and R = X^T Y come from the tcgen05 GEMM
// (fp32 accumulate; ridge_gram in fill_tc.cu). G is then factorised in place as
// L L^T (blocked right-looking Cholesky in fp32, 64 x 64 tiles: the diagonal tile
// in one CTA's shared memory, the panel below it by substitution, the trailing
// lower triangle updated tile by tile), and W = L^-T L^-1 R is solved in place in
// the output by block forward and backward substitution: each 64-row block
// multiplied by its diagonal tile's inverse (all 64 x 64 inverses computed at
// once after the factorisation, so a block's solve is a product with no
// dependent steps), the rest of the right-hand sides updated on the tensor cores
// (the same GEMM, fp32 operands split into bf16 high and low parts).
#include "common.cuh"

namespace tee {

size_t ridge_gram_ws_bytes(int n, int d, int d_out);
tee_status ridge_update_tc(int M, int N, int k3, const void* a3, const void* b3, float* c, int64_t ldc, void* ws,
                           cudaStream_t s);
tee_status ridge_gram(int n, int d, int d_out, const void* x, int64_t ld_x, const void* y, int64_t ld_y, float lambda,
                      float* g, float* r, int64_t ld_r, char* scratch, void* ws, cudaStream_t s);

namespace {

constexpr int NB = 64;           // tile
constexpr int NT = 256;          // threads of the tile kernels
constexpr int TLD = NB + 1;      // shared-memory row stride of a tile (conflict-free columns)

// Factor the diagonal tile k of G (lower triangle) in shared memory. A pivot that
// is not positive records TEE_DEVERR_NOT_SPD with its column and leaves NaN.
__global__ void __launch_bounds__(NT) potrf_tile_kernel(float* __restrict__ G, int64_t ld, int k, void* ws) {
    __shared__ float t[NB][TLD];
    float* base = G + static_cast<int64_t>(k) * NB * ld + static_cast<int64_t>(k) * NB;
    for (int e = threadIdx.x; e < NB * NB; e += NT) t[e / NB][e % NB] = base[static_cast<int64_t>(e / NB) * ld + e % NB];
    __syncthreads();
    for (int j = 0; j < NB; ++j) {
        if (threadIdx.x == 0) {
            const float p = t[j][j];
            if (!(p > 0.f)) record_fault(ws, TEE_DEVERR_NOT_SPD, k * NB + j);
            t[j][j] = sqrtf(p);   // NaN for a pivot <= 0, which then spreads to the solution
        }
        __syncthreads();
        const float dj = t[j][j];
        for (int i = j + 1 + threadIdx.x; i < NB; i += NT) t[i][j] /= dj;
        __syncthreads();
        // trailing update of the tile's lower triangle: t[i][c] -= t[i][j] t[c][j], j < c <= i
        for (int i = j + 1 + (threadIdx.x >> 4); i < NB; i += NT / 16)
            for (int c = j + 1 + (threadIdx.x & 15); c <= i; c += 16) t[i][c] -= t[i][j] * t[c][j];
        __syncthreads();
    }
    for (int e = threadIdx.x; e < NB * NB; e += NT) {
        const int i = e / NB, c = e % NB;
        base[static_cast<int64_t>(i) * ld + c] = c <= i ? t[i][c] : 0.f;
    }
}

// Panel below the diagonal tile k: 16-row slice blockIdx.x % 4 of block row
// i = k + 1 + blockIdx.x / 4 becomes A_ik L_kk^-T (each row solved forward over the
// columns, its dot products split over 16 threads).
constexpr int RPC = 16;   // rows (or right-hand-side columns) per CTA, 16 threads each
__global__ void __launch_bounds__(NT) trsm_panel_kernel(float* __restrict__ G, int64_t ld, int k) {
    __shared__ float l[NB][TLD];
    __shared__ float a[RPC][TLD];
    const int i = k + 1 + blockIdx.x / (NB / RPC), r0 = (blockIdx.x % (NB / RPC)) * RPC;
    const float* lk = G + static_cast<int64_t>(k) * NB * ld + static_cast<int64_t>(k) * NB;
    float* ai = G + (static_cast<int64_t>(i) * NB + r0) * ld + static_cast<int64_t>(k) * NB;
    for (int e = threadIdx.x; e < NB * NB; e += NT) l[e / NB][e % NB] = lk[static_cast<int64_t>(e / NB) * ld + e % NB];
    for (int e = threadIdx.x; e < RPC * NB; e += NT) a[e / NB][e % NB] = ai[static_cast<int64_t>(e / NB) * ld + e % NB];
    __syncthreads();
    const int row = threadIdx.x >> 4, sub = threadIdx.x & 15;   // 16 rows x 16 threads
    for (int c = 0; c < NB; ++c) {
        float s = 0.f;
        for (int cc = sub; cc < c; cc += 16) s = fmaf(a[row][cc], l[c][cc], s);
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (sub == 0) a[row][c] = (a[row][c] - s) / l[c][c];
        __syncwarp();
    }
    __syncthreads();
    for (int e = threadIdx.x; e < RPC * NB; e += NT) ai[static_cast<int64_t>(e / NB) * ld + e % NB] = a[e / NB][e % NB];
}

// C -= A B^T on one 64 x 64 tile, K = 64, fp32; 16 outputs a thread.
__device__ __forceinline__ void tile_update(float* __restrict__ C, int64_t ldc, const float* __restrict__ A,
                                            int64_t lda, const float* __restrict__ B, int64_t ldb,
                                            float (&sa)[NB][TLD], float (&sb)[NB][TLD]) {
    // sa[kk][m] = A(m, kk), sb[kk][c] = B(c, kk)
    for (int e = threadIdx.x; e < NB * NB; e += NT) {
        const int r = e / NB, c = e % NB;
        sa[c][r] = A[static_cast<int64_t>(r) * lda + c];
        sb[c][r] = B[static_cast<int64_t>(r) * ldb + c];
    }
    __syncthreads();
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    float acc[4][4] = {};
#pragma unroll 8
    for (int kk = 0; kk < NB; ++kk) {
        float av[4], bv[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            av[q] = sa[kk][ty * 4 + q];
            bv[q] = sb[kk][tx * 4 + q];
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int w = 0; w < 4; ++w) acc[q][w] = fmaf(av[q], bv[w], acc[q][w]);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int w = 0; w < 4; ++w) C[static_cast<int64_t>(ty * 4 + q) * ldc + tx * 4 + w] -= acc[q][w];
}

// Trailing lower triangle after panel k: tile (i, j), k < j <= i, gets -= L_ik L_jk^T.
__global__ void __launch_bounds__(NT) syrk_kernel(float* __restrict__ G, int64_t ld, int k, int nb) {
    __shared__ float sa[NB][TLD];
    __shared__ float sb[NB][TLD];
    // blockIdx.x -> (i, j) over the lower triangle of the trailing tiles, row by row
    int e = blockIdx.x, i = 0;
    while (e > i) {
        e -= i + 1;
        ++i;
    }
    const int j = e;   // 0 <= j <= i
    const int ti = k + 1 + i, tj = k + 1 + j;
    if (ti >= nb) return;
    float* c = G + static_cast<int64_t>(ti) * NB * ld + static_cast<int64_t>(tj) * NB;
    const float* a = G + static_cast<int64_t>(ti) * NB * ld + static_cast<int64_t>(k) * NB;
    const float* b = G + static_cast<int64_t>(tj) * NB * ld + static_cast<int64_t>(k) * NB;
    tile_update(c, ld, a, ld, b, ld, sa, sb);
}

// The inverse of every diagonal tile of L at once (after the factorisation): CTA
// k inverts L_kk into Li[k] ([64][64], lower triangular) by forward substitution
// on the identity's columns, one column per thread (the columns are independent).
__global__ void __launch_bounds__(NT) trtri_tiles_kernel(const float* __restrict__ G, int64_t ld, float* __restrict__ Li) {
    __shared__ float l[NB][TLD];
    __shared__ float x[NB][TLD];   // x[i][j]: row i of the inverse's column j
    const int k = blockIdx.x;
    const float* lk = G + static_cast<int64_t>(k) * NB * ld + static_cast<int64_t>(k) * NB;
    for (int e = threadIdx.x; e < NB * NB; e += NT) l[e / NB][e % NB] = lk[static_cast<int64_t>(e / NB) * ld + e % NB];
    __syncthreads();
    const int j = threadIdx.x;
    if (j < NB) {
        for (int i = 0; i < j; ++i) x[i][j] = 0.f;
        for (int i = j; i < NB; ++i) {
            float sum = i == j ? 1.f : 0.f;
            for (int c = j; c < i; ++c) sum = fmaf(-l[i][c], x[c][j], sum);
            x[i][j] = sum / l[i][i];
        }
    }
    __syncthreads();
    float* out = Li + static_cast<int64_t>(k) * NB * NB;
    for (int e = threadIdx.x; e < NB * NB; e += NT) out[e] = x[e / NB][e % NB];
}

// fp32 -> bf16 split for the tensor-core updates: x = hi + lo with hi = bf16(x) and
// lo = bf16(x - hi), so that a product of two split values keeps ~16 bits. A row of
// the split operand holds 192 bf16: the 64 values' hi, lo, hi ("A form") or hi,
// hi, lo ("B form"); A-form times B-form summed over the 192 gives
// a_hi b_hi + a_lo b_hi + a_hi b_lo.
constexpr int K3 = 3 * NB;
__device__ __forceinline__ void split_store(__nv_bfloat16* row, int kk, float x, bool b_form) {
    const __nv_bfloat16 hi = __float2bfloat16_rn(x);
    const __nv_bfloat16 lo = __float2bfloat16_rn(x - __bfloat162float(hi));
    row[kk] = hi;
    row[NB + kk] = b_form ? hi : lo;
    row[2 * NB + kk] = b_form ? lo : hi;
}
// dst[r] = split(src[r][0..64)) for r < rows (the 64 values of a row, K along the row).
__global__ void __launch_bounds__(NT) split_rows_kernel(const float* __restrict__ src, int64_t ld, int rows,
                                                        __nv_bfloat16* __restrict__ dst, bool b_form) {
    const int64_t total = static_cast<int64_t>(rows) * NB;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(NT) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * NT) {
        const int64_t r = i / NB;
        const int kk = static_cast<int>(i % NB);
        split_store(dst + r * K3, kk, src[r * ld + kk], b_form);
    }
}
// dst[c] = split(src[0..64)[c]) for c < cols (K down the columns of a 64-row block):
// 64 x 64 tiles through shared memory so that reads and writes stay coalesced.
__global__ void __launch_bounds__(NT) split_cols_kernel(const float* __restrict__ src, int64_t ld, int cols,
                                                        __nv_bfloat16* __restrict__ dst, bool b_form) {
    __shared__ float t[NB][TLD];
    const int c0 = blockIdx.x * NB;
    for (int e = threadIdx.x; e < NB * NB; e += NT) {
        const int kk = e / NB, c = e % NB;
        t[kk][c] = c0 + c < cols ? src[static_cast<int64_t>(kk) * ld + c0 + c] : 0.f;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < NB * NB; e += NT) {
        const int c = e / NB, kk = e % NB;
        if (c0 + c < cols) split_store(dst + static_cast<int64_t>(c0 + c) * K3, kk, t[kk][c], b_form);
    }
}

// One block row of a substitution: R_k <- Li_k R_k (forward) or Li_k^T R_k
// (backward) for the 64 columns 64 blockIdx.x .. + 63, in place (each CTA owns its
// columns), plus the B-form split of the result for the trailing update:
// b3[c][0..192) = split(R_k[0..64)[c]).
__global__ void __launch_bounds__(NT) rhs_mul_kernel(const float* __restrict__ Li, float* __restrict__ R, int64_t ldr,
                                                     int k, bool upper, __nv_bfloat16* __restrict__ b3) {
    __shared__ float sa[NB][TLD];   // sa[kk][m] = A(m, kk): A = Li_k, or Li_k^T
    __shared__ float sb[NB][TLD];   // sb[kk][c] = R_k(kk, c)
    const float* lk = Li + static_cast<int64_t>(k) * NB * NB;
    float* rk = R + static_cast<int64_t>(k) * NB * ldr + static_cast<int64_t>(blockIdx.x) * NB;
    for (int e = threadIdx.x; e < NB * NB; e += NT) {
        const int r = e / NB, c = e % NB;
        sa[c][r] = upper ? lk[c * NB + r] : lk[r * NB + c];
        sb[r][c] = rk[static_cast<int64_t>(r) * ldr + c];
    }
    __syncthreads();
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    float acc[4][4] = {};
#pragma unroll 8
    for (int kk = 0; kk < NB; ++kk) {
        float av[4], bv[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            av[q] = sa[kk][ty * 4 + q];
            bv[q] = sb[kk][tx * 4 + q];
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int w = 0; w < 4; ++w) acc[q][w] = fmaf(av[q], bv[w], acc[q][w]);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const int row = ty * 4 + q, col = tx * 4 + w;
            rk[static_cast<int64_t>(row) * ldr + col] = acc[q][w];
            split_store(b3 + (static_cast<int64_t>(blockIdx.x) * NB + col) * K3, row, acc[q][w], true);
        }
}

}  // namespace

}  // namespace tee

using namespace tee;

static size_t split_bytes(int rows) { return round_up(static_cast<size_t>(rows) * K3 * 2, 1024); }

extern "C" size_t tee_ridge_fit_workspace_size(int32_t n, int32_t d, int32_t d_out) {
    if (n <= 0 || d <= 0 || d_out <= 0) return TEE_WS_HEADER_BYTES;
    const size_t gram = ridge_gram_ws_bytes(n, d, d_out), split = split_bytes(d) + split_bytes(d_out);
    // G (then L), the diagonal tiles' inverses, then the Gram's or the splits' scratch
    return TEE_WS_HEADER_BYTES + round_up(static_cast<size_t>(d) * d * 4, 1024) +
           round_up(static_cast<size_t>(d) * NB * 4, 1024) + (gram > split ? gram : split);
}

extern "C" tee_status tee_ridge_fit(int32_t n, int32_t d, int32_t d_out, const void* x, int64_t ld_x, const void* y,
                                    int64_t ld_y, int32_t dtype, float lambda, float* w, int64_t ld_w, void* ws,
                                    size_t ws_bytes, void* stream) {
    if (n <= 0 || d <= 0 || d_out <= 0 || !x || !y || !w) return TEE_ERR_INVALID_ARG;
    if (dtype != TEE_BF16) return TEE_ERR_UNSUPPORTED;
    if (d % 256 || d_out % 256) return TEE_ERR_UNSUPPORTED;   // the GEMM's 256-column tiles
    if (!(lambda >= 0.f) || ld_x < d || ld_y < d_out || ld_w < d_out || (ld_x * 2) % 16 || (ld_y * 2) % 16 ||
        (ld_w * 4) % 16 || !aligned16(x) || !aligned16(y) || !aligned16(w))
        return TEE_ERR_INVALID_ARG;
    if (!ws || ws_bytes < tee_ridge_fit_workspace_size(n, d, d_out)) return TEE_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* base = static_cast<char*>(ws) + TEE_WS_HEADER_BYTES;
    float* g = reinterpret_cast<float*>(base);
    float* li = reinterpret_cast<float*>(base + round_up(static_cast<size_t>(d) * d * 4, 1024));
    char* scratch = reinterpret_cast<char*>(li) + round_up(static_cast<size_t>(d) * NB * 4, 1024);
    tee_status st = ridge_gram(n, d, d_out, x, ld_x, y, ld_y, lambda, g, w, ld_w, scratch, ws, s);
    if (st != TEE_OK) return st;
    const int nb = d / NB, ncol = d_out / NB;
    for (int k = 0; k < nb; ++k) {   // G = L L^T, in place
        potrf_tile_kernel<<<1, NT, 0, s>>>(g, d, k, ws);
        if ((st = launch_status()) != TEE_OK) return st;
        const int m = nb - 1 - k;
        if (m == 0) break;
        trsm_panel_kernel<<<m * (NB / RPC), NT, 0, s>>>(g, d, k);
        if ((st = launch_status()) != TEE_OK) return st;
        syrk_kernel<<<m * (m + 1) / 2, NT, 0, s>>>(g, d, k, nb);
        if ((st = launch_status()) != TEE_OK) return st;
    }
    // The substitutions' trailing updates run on the tensor cores with split operands
    // (the Gram scratch is free by now): a3 [rows][192] from L, b3 [d_out][192] from
    // the solved block row.
    __nv_bfloat16* a3 = reinterpret_cast<__nv_bfloat16*>(scratch);
    __nv_bfloat16* b3 = reinterpret_cast<__nv_bfloat16*>(scratch + split_bytes(d));
    auto blocks_for = [](int64_t elems) {
        const int64_t b = (elems + NT - 1) / NT;
        return static_cast<int>(b < 2048 ? b : 2048);
    };
    trtri_tiles_kernel<<<nb, NT, 0, s>>>(g, d, li);
    if ((st = launch_status()) != TEE_OK) return st;
    for (int k = 0; k < nb; ++k) {   // L Z = R
        rhs_mul_kernel<<<ncol, NT, 0, s>>>(li, w, ld_w, k, false, b3);   // Z_k = L_kk^-1 R_k, and its split
        if ((st = launch_status()) != TEE_OK) return st;
        const int m = d - (k + 1) * NB;   // rows below: R_i -= L_ik Z_k
        if (m > 0) {
            split_rows_kernel<<<blocks_for(static_cast<int64_t>(m) * NB), NT, 0, s>>>(
                g + static_cast<int64_t>(k + 1) * NB * d + static_cast<int64_t>(k) * NB, d, m, a3, false);
            if ((st = launch_status()) != TEE_OK) return st;
            st = ridge_update_tc(m, d_out, K3, a3, b3, w + static_cast<int64_t>(k + 1) * NB * ld_w, ld_w, ws, s);
            if (st != TEE_OK) return st;
        }
    }
    for (int k = nb - 1; k >= 0; --k) {   // L^T W = Z
        rhs_mul_kernel<<<ncol, NT, 0, s>>>(li, w, ld_w, k, true, b3);   // W_k = L_kk^-T Z_k, and its split
        if ((st = launch_status()) != TEE_OK) return st;
        const int m = k * NB;   // rows above: R_i -= L_ki^T W_k, A[i][kk] = L[k NB + kk][i]
        if (m > 0) {
            split_cols_kernel<<<(m + NB - 1) / NB, NT, 0, s>>>(g + static_cast<int64_t>(k) * NB * d, d, m, a3, false);
            if ((st = launch_status()) != TEE_OK) return st;
            st = ridge_update_tc(m, d_out, K3, a3, b3, w, ld_w, ws, s);
            if (st != TEE_OK) return st;
        }
    }
    return TEE_OK;
}
