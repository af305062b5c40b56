// Exit gate: River-LLM's state-transition cosine and TIDE's RMSNorm router.
//
// Cosine (River-LLM, background "state transition similarity"; method step 3):
// h_prev and h_cur stream in with 128-bit loads, <a,b>, |a|^2 and |b|^2 are
// accumulated in fp32 and reduced with __shfl_xor_sync: one block per token up
// to 1024 tokens (decode batches), one warp per token beyond.
//
// Router (TIDE formula 3; module 4 "Fused LayerNorm + Route"): the d -> b
// contraction is split over (token tile, channel group) blocks that stage the
// token rows in shared memory as fp32; a finalize kernel then applies the
// per-token 1/rms, b_down, SiLU, the b -> 1 projection and the sigmoid. Large
// batches take the tensor-core path in router_tc.cu instead.
//
// Both end in the same decision, score > threshold in fp32, and the same
// "last block" reduction of the all-tokens flag (River-LLM's min over the
// batch; TIDE module 3's "for every token in the batch").
#include <mutex>
#include <type_traits>

#include "common.cuh"

namespace tee {

namespace {

constexpr int GATE_WARPS = 8;
constexpr int GATE_MAX_BLOCKS = 1024;

// 16 bytes of a row that is read once: not kept in L1.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
// <a,b>, |a|^2, |b|^2 over the elements of one 16-byte chunk of each row.
template <typename T>
__device__ __forceinline__ void cos_acc16(uint4 a, uint4 b, float& dot, float& na, float& nb) {
    const uint32_t ua[4] = {a.x, a.y, a.z, a.w}, ub[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        if constexpr (sizeof(T) == 4) {
            const float x = __uint_as_float(ua[q]), y = __uint_as_float(ub[q]);
            dot = fmaf(x, y, dot);
            na = fmaf(x, x, na);
            nb = fmaf(y, y, nb);
        } else {
            float x0, x1, y0, y1;
            if constexpr (std::is_same<T, __half>::value) {
                unpack_f16x2(ua[q], x0, x1);
                unpack_f16x2(ub[q], y0, y1);
            } else {
                unpack_bf16x2(ua[q], x0, x1);
                unpack_bf16x2(ub[q], y0, y1);
            }
            dot = fmaf(x0, y0, dot);
            dot = fmaf(x1, y1, dot);
            na = fmaf(x0, x0, na);
            na = fmaf(x1, x1, na);
            nb = fmaf(y0, y0, nb);
            nb = fmaf(y1, y1, nb);
        }
    }
}

// Large batches: one warp per token, eight 16-byte chunks of each row per lane
// in flight at once (4 KB per row per warp), loads that bypass L1.
constexpr int COS_U = 8;
template <typename T>
__global__ void __launch_bounds__(GATE_WARPS * 32, 3)   // room for the 16 loads in flight
cosine_gate_kernel(int n, int d, const T* __restrict__ hc, int64_t ldc, const T* __restrict__ hp,
                   int64_t ldp, float thr, int rule, bool need_flag, float* __restrict__ score,
                   uint8_t* __restrict__ mask, int32_t* __restrict__ flag, void* ws) {
    allow_dependents();
    constexpr int V = 16 / sizeof(T);   // elements per chunk
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float wmin = INFINITY;
    for (int t = blockIdx.x * GATE_WARPS + warp; t < n; t += gridDim.x * GATE_WARPS) {
        const T* a = hp + static_cast<int64_t>(t) * ldp;
        const T* b = hc + static_cast<int64_t>(t) * ldc;
        float dot = 0.f, na = 0.f, nb = 0.f;
        int i0 = lane * V;
        for (; i0 + (COS_U - 1) * 32 * V < d; i0 += COS_U * 32 * V) {   // whole steps
            uint4 xa[COS_U], xb[COS_U];
#pragma unroll
            for (int u = 0; u < COS_U; ++u) {
                xa[u] = ld_stream16(a + i0 + u * 32 * V);
                xb[u] = ld_stream16(b + i0 + u * 32 * V);
            }
#pragma unroll
            for (int u = 0; u < COS_U; ++u) cos_acc16<T>(xa[u], xb[u], dot, na, nb);
        }
        for (; i0 < d; i0 += 32 * V) cos_acc16<T>(ld_stream16(a + i0), ld_stream16(b + i0), dot, na, nb);   // the rest
        dot = warp_sum(dot);
        na = warp_sum(na);
        nb = warp_sum(nb);
        const float den = sqrtf(na) * sqrtf(nb);
        const float s = den > 0.f ? dot / den : 0.f;
        if (lane == 0) {
            score[t] = s;
            if (rule == TEE_RULE_PER_TOKEN) mask[t] = exits(s, thr);
        }
        wmin = fminf(wmin, s == s ? s : -INFINITY);
    }
    if (!need_flag) return;
    __shared__ float s_min[GATE_WARPS];
    if (lane == 0) s_min[warp] = wmin;
    __syncthreads();
    float bmin = INFINITY;
    if (threadIdx.x == 0)
        for (int w = 0; w < GATE_WARPS; ++w) bmin = fminf(bmin, s_min[w]);
    batch_flag_tail(bmin, n, thr, rule, mask, flag, ws_at<float>(ws, TEE_WS_HEADER_BYTES),
                    ws_counter(ws, WS_CNT_GATE));
}

// Small batches: one block per token, the row split over the block's eight warps,
// so that a decode batch of tens of tokens still spreads over as many SMs and
// each thread issues its loads of both rows at once.
template <typename T>
__global__ void __launch_bounds__(GATE_WARPS * 32)
cosine_gate_row_kernel(int n, int d, const T* __restrict__ hc, int64_t ldc, const T* __restrict__ hp, int64_t ldp,
                       float thr, int rule, bool need_flag, float* __restrict__ score, uint8_t* __restrict__ mask,
                       int32_t* __restrict__ flag, void* ws) {
    allow_dependents();
    const int t = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const T* a = hp + static_cast<int64_t>(t) * ldp;
    const T* b = hc + static_cast<int64_t>(t) * ldc;
    float dot = 0.f, na = 0.f, nb = 0.f;
    for (int i0 = threadIdx.x * 8; i0 < d; i0 += 2 * GATE_WARPS * 32 * 8) {
        float x[2][8], y[2][8];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int i = i0 + u * GATE_WARPS * 32 * 8;
            if (i < d) {
                load8(a + i, x[u]);
                load8(b + i, y[u]);
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) x[u][k] = y[u][k] = 0.f;
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                dot = fmaf(x[u][k], y[u][k], dot);
                na = fmaf(x[u][k], x[u][k], na);
                nb = fmaf(y[u][k], y[u][k], nb);
            }
    }
    __shared__ float s_part[3][GATE_WARPS];
    dot = warp_sum(dot);
    na = warp_sum(na);
    nb = warp_sum(nb);
    if (lane == 0) {
        s_part[0][warp] = dot;
        s_part[1][warp] = na;
        s_part[2][warp] = nb;
    }
    __syncthreads();
    float s = 0.f;
    if (threadIdx.x == 0) {
        dot = na = nb = 0.f;
        for (int w = 0; w < GATE_WARPS; ++w) {
            dot += s_part[0][w];
            na += s_part[1][w];
            nb += s_part[2][w];
        }
        const float den = sqrtf(na) * sqrtf(nb);
        s = den > 0.f ? dot / den : 0.f;
        score[t] = s;
        if (rule == TEE_RULE_PER_TOKEN) mask[t] = exits(s, thr);
        s = s == s ? s : -INFINITY;
    }
    if (!need_flag) return;
    batch_flag_tail(s, n, thr, rule, mask, flag, ws_at<float>(ws, TEE_WS_HEADER_BYTES), ws_counter(ws, WS_CNT_GATE));
}

// ---------------------------------------------------------------- router
constexpr int RT_TOK = 4;        // tokens per block
constexpr int RT_CH_WARP = 1;    // channels per warp
constexpr int RT_WARPS = 8;

// dots[t][c] = sum_i w_down[c][i] * gamma[i] * h[t][i]; sumsq[t] = sum_i h[t][i]^2.
template <typename T>
__global__ void __launch_bounds__(RT_WARPS * 32)
router_dot_kernel(int n, int d, int b, const T* __restrict__ h, int64_t ldh, const T* __restrict__ gamma,
                  const T* __restrict__ wd, float* __restrict__ dots, float* __restrict__ sumsq) {
    extern __shared__ float s_h[];  // [RT_TOK][d], gamma applied
    const int t0 = blockIdx.x * RT_TOK;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Stage the token rows; the blocks of channel group 0 also report sumsq.
    float ss[RT_TOK];
#pragma unroll
    for (int tt = 0; tt < RT_TOK; ++tt) {
        const int t = t0 + tt;
        ss[tt] = 0.f;
        for (int i = threadIdx.x * 8; i < d; i += blockDim.x * 8) {
            float x[8], g[8];
            if (t < n) {
                load8(h + static_cast<int64_t>(t) * ldh + i, x);
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) x[k] = 0.f;
            }
            if (gamma) {
                load8(gamma + i, g);
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) g[k] = 1.f;
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                ss[tt] = fmaf(x[k], x[k], ss[tt]);
                s_h[tt * d + i + k] = x[k] * g[k];
            }
        }
    }
    __shared__ float s_red[RT_TOK][RT_WARPS];
    if (blockIdx.y == 0) {
#pragma unroll
        for (int tt = 0; tt < RT_TOK; ++tt) {
            const float v = warp_sum(ss[tt]);
            if (lane == 0) s_red[tt][warp] = v;
        }
    }
    __syncthreads();
    if (blockIdx.y == 0 && threadIdx.x < RT_TOK && t0 + threadIdx.x < n) {
        float tot = 0.f;
        for (int w = 0; w < RT_WARPS; ++w) tot += s_red[threadIdx.x][w];
        sumsq[t0 + threadIdx.x] = tot;
    }
    for (int cc = 0; cc < RT_CH_WARP; ++cc) {
        const int c = (blockIdx.y * RT_WARPS + warp) * RT_CH_WARP + cc;
        if (c >= b) break;
        float acc[RT_TOK];
#pragma unroll
        for (int tt = 0; tt < RT_TOK; ++tt) acc[tt] = 0.f;
        const T* wrow = wd + static_cast<int64_t>(c) * d;
        // RT_WB pieces of the row per lane in flight: their loads are issued before
        // any of them is used (one round trip per batch, not per piece)
        constexpr int RT_WB = 4;
        for (int i0 = lane * 8; i0 < d; i0 += 256 * RT_WB) {
            float w[RT_WB][8];
#pragma unroll
            for (int u = 0; u < RT_WB; ++u)
                if (i0 + 256 * u < d) load8(wrow + i0 + 256 * u, w[u]);
#pragma unroll
            for (int u = 0; u < RT_WB; ++u) {
                const int i = i0 + 256 * u;
                if (i >= d) break;
#pragma unroll
                for (int tt = 0; tt < RT_TOK; ++tt) {
                    const float4 x0 = *reinterpret_cast<const float4*>(s_h + tt * d + i);
                    const float4 x1 = *reinterpret_cast<const float4*>(s_h + tt * d + i + 4);
                    acc[tt] = fmaf(w[u][0], x0.x, acc[tt]);
                    acc[tt] = fmaf(w[u][1], x0.y, acc[tt]);
                    acc[tt] = fmaf(w[u][2], x0.z, acc[tt]);
                    acc[tt] = fmaf(w[u][3], x0.w, acc[tt]);
                    acc[tt] = fmaf(w[u][4], x1.x, acc[tt]);
                    acc[tt] = fmaf(w[u][5], x1.y, acc[tt]);
                    acc[tt] = fmaf(w[u][6], x1.z, acc[tt]);
                    acc[tt] = fmaf(w[u][7], x1.w, acc[tt]);
                }
            }
        }
#pragma unroll
        for (int tt = 0; tt < RT_TOK; ++tt) {
            const float v = warp_sum(acc[tt]);
            if (lane == 0 && t0 + tt < n) dots[static_cast<int64_t>(t0 + tt) * b + c] = v;
        }
    }
}

}  // namespace

// p[t] = sigmoid(sum_c w_up[c] * SiLU(dots[t][c] / rms_t + b_down[c]) + b_up),
// rms_t = sqrt(sumsq[t] / d + eps): one warp per token. Shared with the
// tensor-core path, which accumulates into dots/sumsq: both are cleared here
// after use, so that the workspace is ready for the next call.
template <typename T>
__global__ void __launch_bounds__(GATE_WARPS * 32)
router_finalize_kernel(int n, int d, int b, float eps, float* __restrict__ dots,
                       float* __restrict__ sumsq, const float* __restrict__ b_down,
                       const T* __restrict__ w_up, const float* __restrict__ b_up, float thr, int rule,
                       bool need_flag, float* __restrict__ score, uint8_t* __restrict__ mask,
                       int32_t* __restrict__ flag, void* ws) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float wmin = INFINITY;
    constexpr int MAXC = 8;  // channels per lane held in registers (b <= 256)
    for (int t = blockIdx.x * GATE_WARPS + warp; t < n; t += gridDim.x * GATE_WARPS) {
        // Issue every load of this token before using any of them.
        float* row = dots + static_cast<int64_t>(t) * b;
        const float ssq = sumsq[t];
        float u[MAXC], wu[MAXC], bd[MAXC];
#pragma unroll
        for (int j = 0; j < MAXC; ++j) {
            const int c = lane + 32 * j;
            u[j] = c < b ? row[c] : 0.f;
            wu[j] = c < b ? to_f32(w_up[c]) : 0.f;
            bd[j] = (c < b && b_down) ? b_down[c] : 0.f;
        }
        __syncwarp();
#pragma unroll
        for (int j = 0; j < MAXC; ++j)
            if (lane + 32 * j < b) row[lane + 32 * j] = 0.f;   // leave the sums cleared for the next call
        if (lane == 0) sumsq[t] = 0.f;
        const float r = 1.0f / sqrtf(ssq / static_cast<float>(d) + eps);
        float z = 0.f;
#pragma unroll
        for (int j = 0; j < MAXC; ++j) {
            const float x = u[j] * r + bd[j];
            z = fmaf(wu[j], __fdividef(x, 1.0f + __expf(-x)), z);   // SiLU (fast exp and divide: ~1e-6 relative)
        }
        z = warp_sum(z);
        if (b_up) z += b_up[0];
        const float p = __fdividef(1.0f, 1.0f + __expf(-z));
        if (lane == 0) {
            score[t] = p;
            if (rule == TEE_RULE_PER_TOKEN) mask[t] = exits(p, thr);
        }
        wmin = fminf(wmin, p == p ? p : -INFINITY);
    }
    if (!need_flag) return;
    __shared__ float s_min[GATE_WARPS];
    if (lane == 0) s_min[warp] = wmin;
    __syncthreads();
    float bmin = INFINITY;
    if (threadIdx.x == 0)
        for (int w = 0; w < GATE_WARPS; ++w) bmin = fminf(bmin, s_min[w]);
    batch_flag_tail(bmin, n, thr, rule, mask, flag, ws_at<float>(ws, TEE_WS_HEADER_BYTES),
                    ws_counter(ws, WS_CNT_ROUTER));
}

// Router gate for small batches (TIDE formula 3; module 4 "Fused LayerNorm +
// Route") in one launch. CTA (kb, th) takes the 64 inputs [64 kb, 64 kb + 64)
// of tokens [32 th, 32 th + 32): it stages their rows (gamma applied) and adds
// the rows' partial sums of squares, then thread (c, half) forms channel c's
// partial dot products with the tokens of its half (tokens 2 j + half) and adds
// them into the workspace's dots[t][c]; the last CTA to finish (a counter)
// finishes every token: 1/rms, b_down, SiLU, w_up, b_up, sigmoid, threshold,
// the batch flag, and leaves dots and sums of squares cleared for the next call.
constexpr int RS_TOK = 32, RS_K = 64, RS_THREADS = 256, RS_LD = RS_K + 4;
constexpr int RS_MAX_TOKENS = 64;

template <typename T>
__global__ void __launch_bounds__(RS_THREADS)
router_small_kernel(int n, int d, int b, const T* __restrict__ h, int64_t ldh, const T* __restrict__ gamma,
                    const T* __restrict__ wd, float* __restrict__ dots, float* __restrict__ sumsq,
                    const float* __restrict__ b_down, const T* __restrict__ w_up, const float* __restrict__ b_up,
                    float eps, float thr, int rule, bool need_flag, float* __restrict__ score,
                    uint8_t* __restrict__ mask, int32_t* __restrict__ flag, uint32_t* __restrict__ counter) {
    __shared__ __align__(16) float s_h[RS_TOK][RS_LD];
    __shared__ float s_min[RS_THREADS / 32];
    __shared__ int s_last;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int k0 = blockIdx.x * RS_K, t0 = blockIdx.y * RS_TOK;
    const int nt = min(RS_TOK, n - t0);
    {   // rows: eight threads per token row, eight inputs each
        const int tt = tid >> 3, e0 = (tid & 7) * 8;
        float x[8], g[8];
        if (tt < nt) {
            load8(h + static_cast<int64_t>(t0 + tt) * ldh + k0 + e0, x);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = 0.f;
        }
        if (gamma) {
            load8(gamma + k0 + e0, g);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) g[e] = 1.f;
        }
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            ss = fmaf(x[e], x[e], ss);
            s_h[tt][e0 + e] = x[e] * g[e];
        }
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        ss += __shfl_xor_sync(0xffffffffu, ss, 2);
        ss += __shfl_xor_sync(0xffffffffu, ss, 4);
        if ((tid & 7) == 0 && tt < nt) atomicAdd(sumsq + t0 + tt, ss);
    }
    __syncthreads();
    {   // channel c = tid / 2, tokens 2 j + (tid & 1)
        const int c = tid >> 1, half = tid & 1;
        if (c < b) {
            float acc[RS_TOK / 2];
#pragma unroll
            for (int j = 0; j < RS_TOK / 2; ++j) acc[j] = 0.f;
            const T* wr = wd + static_cast<int64_t>(c) * d + k0;
            float w[RS_K / 8][8];
#pragma unroll
            for (int q = 0; q < RS_K / 8; ++q) load8(wr + 8 * q, w[q]);   // the whole slice in flight
#pragma unroll
            for (int q = 0; q < RS_K / 8; ++q)
#pragma unroll
                for (int j = 0; j < RS_TOK / 2; ++j) {
                    const float4 a0 = *reinterpret_cast<const float4*>(&s_h[2 * j + half][8 * q]);
                    const float4 a1 = *reinterpret_cast<const float4*>(&s_h[2 * j + half][8 * q + 4]);
                    float v = acc[j];
                    v = fmaf(w[q][0], a0.x, v);
                    v = fmaf(w[q][1], a0.y, v);
                    v = fmaf(w[q][2], a0.z, v);
                    v = fmaf(w[q][3], a0.w, v);
                    v = fmaf(w[q][4], a1.x, v);
                    v = fmaf(w[q][5], a1.y, v);
                    v = fmaf(w[q][6], a1.z, v);
                    v = fmaf(w[q][7], a1.w, v);
                    acc[j] = v;
                }
#pragma unroll
            for (int j = 0; j < RS_TOK / 2; ++j)
                if (2 * j + half < nt) atomicAdd(dots + static_cast<int64_t>(t0 + 2 * j + half) * b + c, acc[j]);
        }
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned prev = atomicAdd(counter, 1u);
        s_last = prev == gridDim.x * gridDim.y - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // the last CTA: warp w finishes tokens w, w + 8, ... (every load of them issued first)
    float wmin = INFINITY;
    constexpr int MAXC = 4;                                    // channels per lane (b <= 128)
    constexpr int TPW = RS_MAX_TOKENS / (RS_THREADS / 32);     // tokens per warp
    float wu[MAXC], bd[MAXC], u[TPW][MAXC], ssq[TPW];
#pragma unroll
    for (int j = 0; j < MAXC; ++j) {
        const int c = lane + 32 * j;
        wu[j] = c < b ? to_f32(w_up[c]) : 0.f;
        bd[j] = (c < b && b_down) ? b_down[c] : 0.f;
    }
#pragma unroll
    for (int i = 0; i < TPW; ++i) {
        const int t = warp + i * (RS_THREADS / 32);
        ssq[i] = t < n ? __ldcg(sumsq + t) : 0.f;
#pragma unroll
        for (int j = 0; j < MAXC; ++j) {
            const int c = lane + 32 * j;
            u[i][j] = (t < n && c < b) ? __ldcg(dots + static_cast<int64_t>(t) * b + c) : 0.f;
        }
    }
#pragma unroll
    for (int i = 0; i < TPW; ++i) {
        const int t = warp + i * (RS_THREADS / 32);
        if (t >= n) break;   // warp-uniform
#pragma unroll
        for (int j = 0; j < MAXC; ++j)
            if (lane + 32 * j < b) dots[static_cast<int64_t>(t) * b + lane + 32 * j] = 0.f;   // cleared for the next call
        if (lane == 0) sumsq[t] = 0.f;
        const float r = 1.0f / sqrtf(ssq[i] / static_cast<float>(d) + eps);
        float z = 0.f;
#pragma unroll
        for (int j = 0; j < MAXC; ++j) {
            const float x = u[i][j] * r + bd[j];
            z = fmaf(wu[j], __fdividef(x, 1.0f + __expf(-x)), z);   // SiLU
        }
        z = warp_sum(z);
        if (b_up) z += b_up[0];
        const float p = __fdividef(1.0f, 1.0f + __expf(-z));
        if (lane == 0) {
            score[t] = p;
            if (rule == TEE_RULE_PER_TOKEN) mask[t] = exits(p, thr);
        }
        wmin = fminf(wmin, p == p ? p : -INFINITY);
    }
    if (tid == 0) *counter = 0u;
    if (!need_flag) return;
    if (lane == 0) s_min[warp] = wmin;
    __syncthreads();
    float m = tid < RS_THREADS / 32 ? s_min[tid] : INFINITY;
    if (warp == 0) {
        m = warp_min(m);
        if (lane == 0) s_min[0] = m;
    }
    __syncthreads();
    const uint8_t f = (n > 0 && s_min[0] > thr) ? 1 : 0;
    if (tid == 0 && flag) *flag = f;
    if (rule == TEE_RULE_BATCH_ALL)
        for (int t = tid; t < n; t += RS_THREADS) mask[t] = f;
}

// Whole router gate on the tensor cores (router_tc.cu). Returns TEE_ERR_UNSUPPORTED
// when the shape does not fit it, so that the CUDA-core kernels run instead.
tee_status router_gate_tc(int n, int d, int b, int dtype, const void* h, int64_t ldh, const void* gamma,
                          const void* w_down, const float* b_down, const void* w_up, const float* b_up, float eps,
                          float thr, int rule, bool need_flag, float* score, uint8_t* mask, int32_t* flag,
                          float* block_mins, uint32_t* counter, void* ws, size_t ws_off, size_t ws_bytes,
                          cudaStream_t stream);
size_t router_tc_scratch_bytes(int n, int d, int b);
size_t router_tc_scratch_bytes_at(int n, int splits);

static size_t gate_blocks(int n) {
    size_t blocks = (static_cast<size_t>(n) + GATE_WARPS - 1) / GATE_WARPS;
    return blocks < 1 ? 1 : (blocks > GATE_MAX_BLOCKS ? GATE_MAX_BLOCKS : blocks);
}

// Workspace: header | block minima (GATE_MAX_BLOCKS f32) | then either the CUDA-core
// path's dots [n][b] f32 and sumsq [n] f32, or the tensor-core path's partials.
static size_t router_dots_off() { return TEE_WS_HEADER_BYTES + GATE_MAX_BLOCKS * sizeof(float); }
static size_t router_sumsq_off(int n, int b) { return round_up(router_dots_off() + static_cast<size_t>(n) * b * 4, 256); }
static size_t router_core_end(int n, int b) { return round_up(router_sumsq_off(n, b) + static_cast<size_t>(n) * 4, 256); }

template <typename T>
static tee_status run_gate(const tee_gate_desc* g, int n, const void* h_cur, int64_t ld_cur, const void* h_prev,
                           int64_t ld_prev, const void* gamma, const void* w_down, const float* b_down,
                           const void* w_up, const float* b_up, float* score, uint8_t* mask, int32_t* flag,
                           void* ws, size_t ws_bytes, cudaStream_t stream) {
    const bool need_flag = flag != nullptr || g->rule == TEE_RULE_BATCH_ALL;
    const int blocks = static_cast<int>(gate_blocks(n));
    if (g->mode == TEE_GATE_COSINE) {
        if (n >= 1 && n <= GATE_MAX_BLOCKS) {   // one block per token (its score is the block minimum)
            cosine_gate_row_kernel<T><<<n, GATE_WARPS * 32, 0, stream>>>(
                n, g->d, static_cast<const T*>(h_cur), ld_cur, static_cast<const T*>(h_prev), ld_prev, g->threshold,
                g->rule, need_flag, score, mask, flag, ws);
            return launch_status();
        }
        // No more blocks than are resident at once: each warp then streams its
        // tokens back to back instead of a second wave starting late.
        static int per_sm = 0;
        if (per_sm == 0 && (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, cosine_gate_kernel<T>,
                                                                           GATE_WARPS * 32, 0) != cudaSuccess ||
                            per_sm < 1)) {
            (void)cudaGetLastError();
            per_sm = 1;
        }
        const int resident = per_sm * sm_count();
        cosine_gate_kernel<T><<<blocks < resident ? blocks : resident, GATE_WARPS * 32, 0, stream>>>(
            n, g->d, static_cast<const T*>(h_cur), ld_cur, static_cast<const T*>(h_prev), ld_prev, g->threshold,
            g->rule, need_flag, score, mask, flag, ws);
        return launch_status();
    }
    const int b = g->bottleneck;
    float* dots = ws_at<float>(ws, router_dots_off());
    float* sumsq = ws_at<float>(ws, router_sumsq_off(n, b));
    tee_status st = router_gate_tc(n, g->d, b, g->dtype, h_cur, ld_cur, gamma, w_down, b_down, w_up, b_up, g->eps,
                                   g->threshold, g->rule, need_flag, score, mask, flag,
                                   ws_at<float>(ws, TEE_WS_HEADER_BYTES), ws_counter(ws, WS_CNT_ROUTER), ws,
                                   router_dots_off(), ws_bytes, stream);
    if (st != TEE_ERR_UNSUPPORTED) return st;   // the tensor-core kernel did the whole gate
    const size_t es = sizeof(T);
    if (n <= RS_MAX_TOKENS && b <= 128 && g->d % RS_K == 0 && aligned16(h_cur) && (ld_cur * es) % 16 == 0 &&
        aligned16(w_down) && (!gamma || aligned16(gamma))) {
        // one launch; its sums accumulate into dots and sumsq, which start cleared
        st = cuda_status(cudaMemsetAsync(dots, 0, router_core_end(n, b) - router_dots_off(), stream));
        if (st != TEE_OK) return st;
        const dim3 grid(g->d / RS_K, (n + RS_TOK - 1) / RS_TOK);
        router_small_kernel<T><<<grid, RS_THREADS, 0, stream>>>(
            n, g->d, b, static_cast<const T*>(h_cur), ld_cur, static_cast<const T*>(gamma),
            static_cast<const T*>(w_down), dots, sumsq, b_down, static_cast<const T*>(w_up), b_up, g->eps,
            g->threshold, g->rule, need_flag, score, mask, flag, ws_counter(ws, WS_CNT_ROUTER));
        return launch_status();
    }
    {
        dim3 grid((n + RT_TOK - 1) / RT_TOK, (b + RT_WARPS * RT_CH_WARP - 1) / (RT_WARPS * RT_CH_WARP));
        const size_t smem = static_cast<size_t>(RT_TOK) * g->d * sizeof(float);
        if (smem > 48 * 1024) {
            st = cuda_status(cudaFuncSetAttribute(router_dot_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                  static_cast<int>(smem)));
            if (st != TEE_OK) return st;
        }
        router_dot_kernel<T><<<grid, RT_WARPS * 32, smem, stream>>>(
            n, g->d, b, static_cast<const T*>(h_cur), ld_cur, static_cast<const T*>(gamma),
            static_cast<const T*>(w_down), dots, sumsq);
        st = launch_status();
    }
    if (st != TEE_OK) return st;
    router_finalize_kernel<T><<<blocks, GATE_WARPS * 32, 0, stream>>>(
        n, g->d, b, g->eps, dots, sumsq, b_down, static_cast<const T*>(w_up), b_up, g->threshold, g->rule,
        need_flag, score, mask, flag, ws);
    return launch_status();
}

}  // namespace tee

using namespace tee;

// Smallest workspace a call accepts: the router's tensor-core path then splits K
// least (the size asked for by tee_exit_gate_workspace_size lets it split most).
static size_t gate_min_workspace(const tee_gate_desc* g, int n) {
    if (g->mode == TEE_GATE_COSINE) return TEE_WS_HEADER_BYTES + GATE_MAX_BLOCKS * sizeof(float);
    const int b = g->bottleneck > 0 ? g->bottleneck : 128;
    const size_t core = router_core_end(n, b);
    const size_t tc = router_dots_off() + router_tc_scratch_bytes_at(n, 1);
    return core > tc ? core : tc;
}

extern "C" size_t tee_exit_gate_workspace_size(const tee_gate_desc* g, int32_t n) {
    if (!g || n < 0) return 0;
    if (g->mode == TEE_GATE_COSINE) return gate_min_workspace(g, n);
    const int b = g->bottleneck > 0 ? g->bottleneck : 128;
    const size_t core = router_core_end(n, b);
    const size_t tc = router_dots_off() + router_tc_scratch_bytes(n, g->d, b);
    const size_t m = core > tc ? core : tc;
    const size_t lo = gate_min_workspace(g, n);
    return m > lo ? m : lo;
}

extern "C" tee_status tee_exit_gate(const tee_gate_desc* g, int32_t n, const void* h_cur, int64_t ld_cur,
                                    const void* h_prev, int64_t ld_prev, const void* gamma, const void* w_down,
                                    const float* b_down, const void* w_up, const float* b_up, float* score,
                                    uint8_t* mask, int32_t* batch_flag, void* ws, size_t ws_bytes, void* stream) {
    if (!g || n < 0 || g->d <= 0 || g->d % 8 != 0) return TEE_ERR_INVALID_ARG;
    if (g->mode != TEE_GATE_COSINE && g->mode != TEE_GATE_ROUTER) return TEE_ERR_INVALID_ARG;
    if (g->rule != TEE_RULE_PER_TOKEN && g->rule != TEE_RULE_BATCH_ALL) return TEE_ERR_INVALID_ARG;
    if (g->threshold != g->threshold) return TEE_ERR_INVALID_ARG;
    const size_t es = dtype_bytes(g->dtype);
    if (es == 0) return TEE_ERR_UNSUPPORTED;
    if (!ws || ws_bytes < gate_min_workspace(g, n)) return TEE_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (n == 0) {
        if (batch_flag) return cuda_status(cudaMemsetAsync(batch_flag, 0, sizeof(int32_t), s));
        return TEE_OK;
    }
    if (!h_cur || !score || !mask || ld_cur < g->d || !aligned16(h_cur) || (ld_cur * es) % 16) return TEE_ERR_INVALID_ARG;
    if (g->mode == TEE_GATE_COSINE) {
        if (!h_prev || ld_prev < g->d || !aligned16(h_prev) || (ld_prev * es) % 16) return TEE_ERR_INVALID_ARG;
    } else {
        if (!w_down || !w_up || g->bottleneck <= 0 || g->bottleneck > 256 || !aligned16(w_down))
            return TEE_ERR_INVALID_ARG;
        if (gamma && !aligned16(gamma)) return TEE_ERR_INVALID_ARG;
        if (!(g->eps >= 0.f)) return TEE_ERR_INVALID_ARG;
    }
    switch (g->dtype) {
        case TEE_F32:
            return run_gate<float>(g, n, h_cur, ld_cur, h_prev, ld_prev, gamma, w_down, b_down, w_up, b_up, score,
                                   mask, batch_flag, ws, ws_bytes, s);
        case TEE_F16:
            return run_gate<__half>(g, n, h_cur, ld_cur, h_prev, ld_prev, gamma, w_down, b_down, w_up, b_up, score,
                                    mask, batch_flag, ws, ws_bytes, s);
        default:
            return run_gate<__nv_bfloat16>(g, n, h_cur, ld_cur, h_prev, ld_prev, gamma, w_down, b_down, w_up, b_up,
                                           score, mask, batch_flag, ws, ws_bytes, s);
    }
}

// ---------------------------------------------------------------------------
// Router gate without a caller workspace.
//
// Some callers cannot hand the library any device scratch: a plugin whose host
// owns all device memory through its own pool and passes the plugin nothing but
// the call's inputs and outputs, or a latency-critical loop where cudaMalloc is
// ruled out because it can block or synchronise the device. For them the
// router gate can take its scratch (per-token channel sums and sum of squares,
// per-block minima, the last-block counter) from a fixed array compiled into
// the library. Every GPU that loads the library holds this array until the
// process exits.
constexpr size_t ROUTER_STATIC_SCRATCH_BYTES = size_t(4) << 20;  // 4 MiB
static __device__ __align__(256) unsigned char g_router_scratch[ROUTER_STATIC_SCRATCH_BYTES];

constexpr int STATIC_MAX_DEVICES = 64;
static std::mutex g_router_scratch_mu;
static void* g_router_scratch_addr[STATIC_MAX_DEVICES] = {};

// Device address of the array on the current device. Host code only knows a
// host-side stand-in for it, so the address comes from cudaGetSymbolAddress,
// looked up once per device with that device current.
static tee_status router_static_scratch(void** out) {
    int dev = 0;
    tee_status st = cuda_status(cudaGetDevice(&dev));
    if (st != TEE_OK) return st;
    if (dev < 0 || dev >= STATIC_MAX_DEVICES) return TEE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_router_scratch_mu);
    if (!g_router_scratch_addr[dev]) {
        void* p = nullptr;
        st = cuda_status(cudaGetSymbolAddress(&p, g_router_scratch));
        if (st != TEE_OK) return st;
        g_router_scratch_addr[dev] = p;
    }
    *out = g_router_scratch_addr[dev];
    return TEE_OK;
}

extern "C" size_t tee_exit_gate_router_static_max_bytes(void) { return ROUTER_STATIC_SCRATCH_BYTES; }

extern "C" tee_status tee_exit_gate_router_static(const tee_gate_desc* g, int32_t n, const void* h, int64_t ld,
                                                  const void* gamma, const void* w_down, const float* b_down,
                                                  const void* w_up, const float* b_up, float* score,
                                                  uint8_t* mask, int32_t* batch_flag, void* stream) {
    if (!g || g->mode != TEE_GATE_ROUTER) return TEE_ERR_INVALID_ARG;
    if (n < 0) return TEE_ERR_INVALID_ARG;
    const size_t need = gate_min_workspace(g, n);
    if (need > ROUTER_STATIC_SCRATCH_BYTES) return TEE_ERR_WORKSPACE;
    void* scratch = nullptr;
    tee_status st = router_static_scratch(&scratch);
    if (st != TEE_OK) return st;
    // The array keeps the previous call's contents. The last-block counters of
    // the header must start at zero; the fault word (the header's first two
    // words) is sticky, read by tee_exit_gate_router_static_device_error and
    // cleared only by tee_exit_gate_router_static_clear_error.
    constexpr size_t FAULT_BYTES = 2 * sizeof(int32_t);
    st = cuda_status(cudaMemsetAsync(static_cast<unsigned char*>(scratch) + FAULT_BYTES, 0,
                                     TEE_WS_HEADER_BYTES - FAULT_BYTES, static_cast<cudaStream_t>(stream)));
    if (st != TEE_OK) return st;
    return tee_exit_gate(g, n, h, ld, nullptr, 0, gamma, w_down, b_down, w_up, b_up, score, mask, batch_flag,
                         scratch, ROUTER_STATIC_SCRATCH_BYTES, stream);
}

extern "C" tee_status tee_exit_gate_router_static_device_error(int32_t* code, int32_t* detail, void* stream) {
    void* scratch = nullptr;
    tee_status st = router_static_scratch(&scratch);
    if (st != TEE_OK) return st;
    return tee_get_device_error(scratch, code, detail, stream);
}

extern "C" tee_status tee_exit_gate_router_static_clear_error(void* stream) {
    void* scratch = nullptr;
    tee_status st = router_static_scratch(&scratch);
    if (st != TEE_OK) return st;
    return tee_clear_device_error(scratch, stream);
}
