// The Exit River (River-LLM, core method and method steps 1 and 3): the tokens
// that left the backbone run the W4A16 copies of the remaining decoder layers,
// each of which writes the skipped layer's K/V into the backbone's slots.
//
// One call = a prologue kernel and, per exit layer, five launches:
//   river_gather        h rows -> fp32 residual stream, bf16 (h * attn_norm),
//                       sum(h^2) per item; item checks; counters cleared
//   w4_gemm<QKV>        [q|k|v] = (h * g) . [Wq|Wk|Wv], times 1/rms(h); RoPE on
//                       q and k; q to the workspace, k and v to the cache slot
//   river_attn_pair     (or river_attn_split for few items) scores and P.V as
//                       warp-level tensor-core products over TMA-fed K/V
//                       chunks: persistent consumer groups each walking one
//                       (item, kv head) pair's chunks with an online softmax, or
//                       one CTA per chunk whose partials the last chunk merges
//   w4_gemm<O>          h1 = h + o . Wo; bf16 (h1 * ffn_norm) and sum(h1^2)
//   w4_gemm<GU>         gate | up from (h1 * g2) . [Wg|Wu] (64 columns of each
//                       per tile), times 1/rms(h1); a = SiLU(gate) * up (bf16)
//   w4_gemm<DOWN>       h2 = h1 + a . Wd; bf16 (h2 * next attn_norm) and
//                       sum(h2^2), or h_out = bf16(h2) after the last layer
// RMSNorm's row scale commutes out of the contraction: A holds h * g in bf16
// and the epilogue multiplies by 1/rms, whose sum of squares the producing
// kernel accumulated in fp32.
//
// w4_gemm (tcgen05): a CTA computes a 128-column tile for every item (items <=
// 128) over a 1/ks slice of the inputs; the ks CTAs of a tile are one cluster.
// Per stage of two 64-input blocks, one warp brings the packed int4 weights
// (repacked per tile at prepare time) by one bulk copy and another the A tiles
// by one TMA box; two groups of eight warps, on alternate stages, dequantise the
// weights into B tiles; one thread issues the transposed MMAs (M = the 128
// output columns, N = the items rounded up to 16, K = 16) into TMEM. The CTAs
// then reduce their partial tiles through distributed shared memory, each
// finishing its share of the columns with the mode's epilogue.
#include <algorithm>

#include "fill.cuh"
#include "tc.cuh"

namespace tee {

namespace {

using bf16 = __nv_bfloat16;

constexpr uint32_t RIVER_MAGIC = 0x54455256u;  // "TERV"

// ------------------------------------------------------------------ workspace
struct RiverWs {
    size_t resid, abuf, qbuf, obuf, act, ss_a, ss_f, ipos, iseq, acnt, apart, end;
    bool by_pair;   // the attention walks whole (item, kv head) pairs (else chunks, with partials)
};

constexpr int GT_N = 128;        // output columns per GEMM tile
constexpr int GT_K = 64;         // inputs per k block
constexpr int G_DQ_WARPS = 16;   // dequantising warps (then the epilogue)
constexpr int G_PROD_WARP = G_DQ_WARPS;       // issues the weights' bulk copies
constexpr int G_MMA_WARP = G_DQ_WARPS + 1;    // issues the MMAs, owns TMEM
constexpr int G_A_WARP = G_DQ_WARPS + 2;      // issues the A tiles' TMA copies
constexpr int G_THREADS = (G_DQ_WARPS + 3) * 32;
constexpr int G_DQ_GROUPS = 2;   // dequantising groups; group q takes the stages j with j % G_DQ_GROUPS == q
constexpr int G_DQ_GWARPS = G_DQ_WARPS / G_DQ_GROUPS;
constexpr int G_DQ_PARTS = G_DQ_GWARPS * 32 / 128;   // threads per column: each takes 32 / G_DQ_PARTS packed rows
constexpr int G_EPI_THREADS = G_DQ_WARPS * 32;
// A stage = two k blocks (G_BPS). Rings: the packed weights (G_WS stages with
// their own full / empty barriers, released by the dequantising group once it
// has read them), and the A tiles and dequantised B tiles (G_BP stages each, own
// full barriers, one empty barrier per stage that the MMAs' single commit
// releases for both). The MMA is transposed:
// M = the tile's 128 output columns (the dequantised weights), N = the item rows
// (a multiple of 16), so the accumulator holds [column][item], the tensor core
// does no work for absent items and reads no rows past them.
constexpr int G_BPS = 2;         // k blocks per stage
constexpr int G_WS = 3;          // weight stages
constexpr int G_BP = 3;          // A and B stages
constexpr int G_RB = G_BP * G_BPS;   // dequantised B buffers
constexpr int G_A_ROWS = 128;    // A tile rows (the MMA's N) at most
constexpr uint32_t G_A_STAGE = G_BPS * G_A_ROWS * 128;   // 32 KB: two tiles of up to 128 rows
constexpr uint32_t G_A_REGION = G_BP * G_A_STAGE;        // the A ring
constexpr uint32_t G_B_BYTES = GT_N * GT_K * 2;      // 16 KB
// a packed weight block: codes [32 packed rows][128 columns], then 128 fp16 scales, 128 fp16 zeros
constexpr uint32_t G_W_BYTES = 32 * GT_N + 2 * GT_N * 2;   // 4608
constexpr uint32_t G_OFF_A = 0;
constexpr uint32_t G_OFF_B = G_OFF_A + G_A_REGION;
constexpr uint32_t G_OFF_W = G_OFF_B + G_RB * G_B_BYTES;
constexpr uint32_t G_OFF_BAR = G_OFF_W + G_WS * G_BPS * G_W_BYTES;
constexpr size_t G_SMEM = 1024 + G_OFF_BAR + (2 * G_WS + 3 * G_BP + 1) * 8 + 16;
// the CTA's partial tile after the loop: [128 rows][GT_N + 4] fp32, over the B ring
constexpr int G_P_PITCH = GT_N + 4;
static_assert(G_A_ROWS * G_P_PITCH * 4 <= G_RB * G_B_BYTES, "partial tile fits the B ring");
static_assert(G_OFF_B % 1024 == 0 && G_OFF_W % 16 == 0 && G_OFF_BAR % 8 == 0, "alignment");
static_assert(G_SMEM <= 232448, "shared memory");

constexpr int MAX_KS = 8;        // K splits = CTAs of a cluster (portable size)
constexpr int MAX_ITEMS = 128;

constexpr int KG_CNT = 64 * 8;   // counters of the two-cluster K split: tiles (<= 64) x ks (<= 8)
// Attention chunks, one TMA box per 64 columns of K and of V (the last chunk of a
// sequence reads up to a chunk's rows less one that it does not use): 16 KB of K
// for the pair kernel, 32 KB for the split kernel.
__host__ __device__ constexpr int at_pair_box(int hd) { return 8192 / hd; }
__host__ __device__ constexpr int at_split_box(int hd) { return 16384 / hd; }

int max_clusters(int ks);

// K splits (the CTAs of one cluster): the largest power of two that keeps every
// cluster resident at once, tiles * ks within the SMs, and each split at least
// two 64-input blocks.
int choose_ks(int tiles, int K) {
    const int sms = sm_count();
    int ks = 1;
    while (ks * 2 <= MAX_KS && tiles * ks * 2 <= sms && K % (ks * 2 * GT_K) == 0 && K / (ks * 2) >= 2 * GT_K &&
           tiles <= max_clusters(ks * 2))
        ks *= 2;
    return ks;
}

// K groups for the residual GEMMs (O, DOWN): a second cluster of ks CTAs per tile
// when the doubled grid still fits the SMs and each split keeps eight 64-input
// blocks (with fewer, as in the 2048-input o projection, the extra launch width
// costs more than it brings: 13.2 us against 11.8 us measured).
int choose_kg(int tiles, int ks, int K) {
    const int sms = sm_count();
    return (ks >= 2 && tiles * ks * 2 <= sms && tiles * ks <= KG_CNT && K % (ks * 2 * GT_K) == 0 &&
            K / (ks * 2) >= 8 * GT_K)
               ? 2
               : 1;
}

int attn_chunks(const tee_river_desc& D, int max_pos) {
    return (max_pos + at_split_box(D.head_dim) - 1) / at_split_box(D.head_dim);
}
// The split walk's merge keeps 3 floats per (query head of a group, chunk) in the
// 32 KB V buffer of its CTA.
bool split_merge_fits(const tee_river_desc& D, int max_pos) {
    const int rep = D.n_q_heads / std::max(1, D.n_kv_heads);
    return static_cast<size_t>(attn_chunks(D, max_pos)) * rep * 3 * 4 <=
           static_cast<size_t>(at_split_box(D.head_dim)) * D.head_dim * 2;
}
// The pair kernel's consumer groups (two per SM) want a pair each at least; a
// cache too long for the split walk's merge goes to the pair walk too.
bool attn_by_pair(const tee_river_desc& D, int n_max, int max_pos) {
    if (D.flags == TEE_RIVER_ATTN_BY_PAIR) return true;
    if (D.flags == TEE_RIVER_ATTN_BY_CHUNK) return false;
    return static_cast<int64_t>(n_max) * D.n_kv_heads >= static_cast<int64_t>(2) * sm_count() ||
           !split_merge_fits(D, max_pos);
}

RiverWs river_ws(const tee_river_desc& D, int n_max, int max_pos) {
    const size_t n = static_cast<size_t>(n_max > 0 ? n_max : 1);
    const size_t d = D.d, qw = static_cast<size_t>(D.n_q_heads) * D.head_dim, f = D.d_ff;
    const size_t rep = static_cast<size_t>(D.n_q_heads / std::max(1, D.n_kv_heads));
    RiverWs w{};
    size_t o = TEE_WS_HEADER_BYTES;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = round_up(o + bytes, 256);
        return at;
    };
    w.resid = take(n * d * 4);
    const size_t na = G_A_ROWS;   // the GEMMs' A operands: 128 rows, the TMA map's extent
    w.abuf = take(na * d * 2);
    w.qbuf = take(n * qw * 2);
    w.obuf = take(na * qw * 2);
    w.act = take(na * f * 2);
    w.ss_a = take(n * 4);
    w.ss_f = take(n * 4);
    w.ipos = take(n * 4);
    w.iseq = take(n * 4);
    w.by_pair = attn_by_pair(D, n_max, max_pos);
    // the K groups' counters (tiles x ks), then (split attention) the chunks' arrival counters
    w.acnt = take((KG_CNT + (w.by_pair ? 0 : n * D.n_kv_heads)) * 4);
    w.apart = w.by_pair ? 0 : take(n * D.n_kv_heads * attn_chunks(D, max_pos) * rep * (D.head_dim + 2) * 4);
    w.end = o;
    return w;
}

// ------------------------------------------------------------------ prologue
struct GatherArgs {
    int n_max;
    const int32_t* n_dev;
    const bf16* h;
    int64_t ld_h;
    int h_rows;
    const int32_t* rows;
    const int32_t* pos;
    const int32_t* seq;
    tee_cache_layout cl;
    const PrepHeader* hdr;
    int d;
    const bf16* gain;
    float* resid;
    bf16* abuf;
    float* ss_a;
    float* ss_f;
    int32_t* ipos;
    int32_t* iseq;
    int32_t* cnt;   // the arrival counters (K-split GEMMs, split attention)
    int n_cnt;
};

__global__ void __launch_bounds__(256) river_gather_kernel(GatherArgs a, void* ws) {
    allow_dependents();
    const int m = blockIdx.x;
    if (m == 0)
        for (int i = threadIdx.x; i < a.n_cnt; i += blockDim.x) a.cnt[i] = 0;
    const int n = item_count(a.n_max, a.n_dev);
    if (m >= n) return;
    __shared__ float s_red[8];
    __shared__ int s_ok;
    if (threadIdx.x == 0) {
        int ok = 1;
        const int r = a.rows ? a.rows[m] : m;
        int p = -1, s = 0;
        if (r < 0 || r >= a.h_rows) {
            record_fault(ws, TEE_DEVERR_ROW, r);
            ok = 0;
        } else {
            p = a.pos[r];
            s = a.seq ? a.seq[r] : 0;
            if (!pos_ok(p, a.cl.max_pos, a.hdr)) {
                record_fault(ws, TEE_DEVERR_POS, p);
                ok = 0;
            } else if (s < 0 || s >= a.cl.n_seq) {
                record_fault(ws, TEE_DEVERR_SEQ, s);
                ok = 0;
            }
        }
        a.ipos[m] = ok ? p : -1;
        a.iseq[m] = ok ? s : 0;
        s_ok = ok ? r : -1;
    }
    __syncthreads();
    const int r = s_ok;
    float ss = 0.f;
    float* res = a.resid + static_cast<int64_t>(m) * a.d;
    bf16* ab = a.abuf + static_cast<int64_t>(m) * a.d;
    for (int k = threadIdx.x * 8; k < a.d; k += blockDim.x * 8) {
        float x[8], g[8];
        if (r >= 0) {
            load8(a.h + static_cast<int64_t>(r) * a.ld_h + k, x);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = 0.f;
        }
        load8(a.gain + k, g);
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
#pragma unroll
        for (int e = 0; e < 4; ++e) o[e] = pack_bf16x2(x[2 * e] * g[2 * e], x[2 * e + 1] * g[2 * e + 1]);
        *reinterpret_cast<float4*>(res + k) = make_float4(x[0], x[1], x[2], x[3]);
        *reinterpret_cast<float4*>(res + k + 4) = make_float4(x[4], x[5], x[6], x[7]);
        *reinterpret_cast<uint4*>(ab + k) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) t += s_red[w];
        a.ss_a[m] = t;
        a.ss_f[m] = 0.f;
    }
}

// ------------------------------------------------------------------ W4A16 GEMM
enum { M_QKV = 0, M_O = 1, M_GU = 2, M_DOWN = 3 };

struct W4Seg {
    const uint8_t* codes;   // [K/2][n]
    const __half* scale;    // [K/64][n]
    const __half* zero;
    int n;
};

struct GemmArgs {
    CUtensorMap tm_a;       // A [128][K] bf16 as K/64 blocks, box 2 blocks x a_rows x 64, 128-byte swizzle
    const uint8_t* blob;    // packed weights [tile][K/64][G_W_BYTES]
    int K, N, ks;
    // K groups: kg clusters of ks CTAs per tile, each over 1/kg of K (O and DOWN only);
    // with kg = 2 both add their sums into the residual and the second to arrive
    // (kg_cnt[tile][rank], zero between calls) finishes the tile's columns
    int kg;
    int32_t* kg_cnt;
    int n_max;
    const int32_t* n_dev;
    const bf16* a;          // [128][lda]
    int64_t lda;
    int a_rows;             // rows of A that TMA brings = the MMA's N (the item bound rounded up to 16;
                            // rows past the items feed only accumulator columns that are never read)
    float* ss_zero;         // cleared by CTA (0, 0): the next producer accumulates into it
    // row scale of the normalised input: rs = 1 / sqrt(ss_in / width + eps)
    const float* ss_in;
    float inv_width, eps;
    // QKV
    int qw, kvw, hd, half;
    bf16* qbuf;
    const int32_t* ipos;
    const int32_t* iseq;
    const float2* rope;
    bf16* kc;
    bf16* vc;
    tee_cache_layout cl;
    int layer;
    // O / DOWN: residual update, the next normalised input (or the output)
    float* resid;
    int d;
    const bf16* next_gain;
    bf16* next_a;
    float* ss_out;
    bf16* h_out;
    int64_t ld_out;
    // GU
    bf16* act;
    int d_ff;
};

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(tc::smem_u32(dst)), "l"(src), "r"(bytes), "r"(tc::smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ float row_scale(const GemmArgs& g, int m) {
    return g.ss_in ? 1.0f / sqrtf(g.ss_in[m] * g.inv_width + g.eps) : 1.f;
}

__device__ __forceinline__ uint2 pack4_bf16(float a, float b, float c, float d) {
    return make_uint2(pack_bf16x2(a, b), pack_bf16x2(c, d));
}

__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// Sum over the cluster's ks partial tiles of (row m, columns col .. col + 3), in
// rank order; every CTA's load is issued before the first add.
__device__ __forceinline__ float4 tile_sum4(const float* P, int ks, int m, int col) {
    const uint32_t laddr = tc::smem_u32(P + m * G_P_PITCH + col);
    if (ks == 1) return *reinterpret_cast<const float4*>(P + m * G_P_PITCH + col);
    float4 v[MAX_KS];
#pragma unroll
    for (int r = 0; r < MAX_KS; ++r)
        if (r < ks) {
            uint32_t ra;
            asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(laddr), "r"(r));
            asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(v[r].x), "=f"(v[r].y), "=f"(v[r].z), "=f"(v[r].w)
                         : "r"(ra)
                         : "memory");
        }
    float4 a = v[0];
#pragma unroll
    for (int r = 1; r < MAX_KS; ++r)
        if (r < ks) {
            a.x += v[r].x;
            a.y += v[r].y;
            a.z += v[r].z;
            a.w += v[r].w;
        }
    return a;
}

__device__ __forceinline__ void finish_residual(const GemmArgs& g, float4 v, int m, int col, int gpr);

// The tile's epilogue for this CTA's share of it (groups [rank * gpr, (rank + 1) * gpr)
// of four consecutive columns, pairs or units); a thread takes one group of one item.
template <int MODE>
__device__ void finish_tile(const GemmArgs& g, const float* P, int t, int n, int rank) {
    const int tid = threadIdx.x;
    const int c0 = t * GT_N;
    constexpr int G = MODE == M_QKV || MODE == M_GU ? 16 : 32;   // groups per tile
    const int gpr = G / g.ks;
    for (int idx = tid; idx < n * gpr; idx += G_EPI_THREADS) {
        const int m = idx / gpr, grp = rank * gpr + idx % gpr;
        if (MODE == M_QKV) {
            const int p = 4 * grp;   // four pairs (i, i + half)
            const int ht = p / g.half, i = p % g.half;
            const int lo = ht * g.hd + i, hi = lo + g.half;   // tile columns
            const int pm = g.ipos[m];
            if (pm < 0) continue;
            const float rs = row_scale(g, m);
            const float4 a = tile_sum4(P, g.ks, m, lo), b = tile_sum4(P, g.ks, m, hi);
            float x1[4] = {a.x * rs, a.y * rs, a.z * rs, a.w * rs}, x2[4] = {b.x * rs, b.y * rs, b.z * rs, b.w * rs};
            const int glo = c0 + lo;
            const bool is_v = glo >= g.qw + g.kvw;
            if (!is_v) {
                const float4* cs = reinterpret_cast<const float4*>(g.rope + static_cast<int64_t>(pm) * g.half + i);
                const float4 e01 = cs[0], e23 = cs[1];
                const float c[4] = {e01.x, e01.z, e23.x, e23.z}, sn[4] = {e01.y, e01.w, e23.y, e23.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float y1 = x1[e] * c[e] - x2[e] * sn[e], y2 = x2[e] * c[e] + x1[e] * sn[e];
                    x1[e] = y1;
                    x2[e] = y2;
                }
            }
            const uint2 plo = pack4_bf16(x1[0], x1[1], x1[2], x1[3]), phi = pack4_bf16(x2[0], x2[1], x2[2], x2[3]);
            bf16* dst;
            if (glo < g.qw) {
                dst = g.qbuf + static_cast<int64_t>(m) * g.qw + glo;
            } else {
                const int cc = is_v ? glo - g.qw - g.kvw : glo - g.qw;
                dst = (is_v ? g.vc : g.kc) + g.layer * g.cl.s_layer + g.iseq[m] * g.cl.s_seq +
                      (cc / g.hd) * g.cl.s_head + static_cast<int64_t>(pm) * g.cl.s_pos + cc % g.hd;
            }
            *reinterpret_cast<uint2*>(dst) = plo;
            *reinterpret_cast<uint2*>(dst + g.half) = phi;
        } else if (MODE == M_GU) {
            const int u = 4 * grp;
            const float rs = row_scale(g, m);
            const float4 ga = tile_sum4(P, g.ks, m, u), up = tile_sum4(P, g.ks, m, 64 + u);
            const float gv[4] = {ga.x * rs, ga.y * rs, ga.z * rs, ga.w * rs};
            const float uv[4] = {up.x * rs, up.y * rs, up.z * rs, up.w * rs};
            float a[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) a[e] = gv[e] / (1.0f + expf(-gv[e])) * uv[e];
            *reinterpret_cast<uint2*>(g.act + static_cast<int64_t>(m) * g.d_ff + 64 * t + u) =
                pack4_bf16(a[0], a[1], a[2], a[3]);
        } else {   // M_O, M_DOWN: residual update
            const int lc = 4 * grp, col = c0 + lc;
            float4* rp = reinterpret_cast<float4*>(g.resid + static_cast<int64_t>(m) * g.d + col);
            const float4 sum = tile_sum4(P, g.ks, m, lc);
            if (g.kg > 1) {   // the other K group adds its part too; the second to arrive finishes below
                atomicAdd(&rp->x, sum.x);
                atomicAdd(&rp->y, sum.y);
                atomicAdd(&rp->z, sum.z);
                atomicAdd(&rp->w, sum.w);
                continue;
            }
            float4 v = *rp;
            v.x += sum.x;
            v.y += sum.y;
            v.z += sum.z;
            v.w += sum.w;
            *rp = v;
            finish_residual(g, v, m, col, gpr);
        }
    }
    if ((MODE == M_O || MODE == M_DOWN) && g.kg > 1) {
        // both K groups' sums are in the residual once the second group's CTA of this
        // rank arrives: it writes the next normalised input (or the output)
        __shared__ int s_second;
        __threadfence();
        asm volatile("bar.sync 1, %0;" ::"r"(G_EPI_THREADS) : "memory");
        if (tid == 0) {
            int32_t* ctr = g.kg_cnt + t * g.ks + rank;
            const int prev = atomicAdd(ctr, 1);
            s_second = prev == g.kg - 1;
            if (s_second) *ctr = 0;
        }
        asm volatile("bar.sync 1, %0;" ::"r"(G_EPI_THREADS) : "memory");
        if (!s_second) return;
        __threadfence();
        for (int idx = tid; idx < n * gpr; idx += G_EPI_THREADS) {
            const int m = idx / gpr, col = c0 + 4 * (rank * gpr + idx % gpr);
            const float4 v = __ldcg(reinterpret_cast<const float4*>(g.resid + static_cast<int64_t>(m) * g.d + col));
            finish_residual(g, v, m, col, gpr);
        }
    }
}

// After the residual update of (item m, columns col .. col + 3): the output row
// (last layer), or the next normalised input and its sum of squares.
__device__ __forceinline__ void finish_residual(const GemmArgs& g, float4 v, int m, int col, int gpr) {
    if (g.h_out) {
        if (g.ipos[m] >= 0)
            *reinterpret_cast<uint2*>(g.h_out + static_cast<int64_t>(m) * g.ld_out + col) = pack4_bf16(v.x, v.y, v.z, v.w);
        return;
    }
    const uint2 gg = *reinterpret_cast<const uint2*>(g.next_gain + col);
    float g0, g1, g2, g3;
    unpack_bf16x2(gg.x, g0, g1);
    unpack_bf16x2(gg.y, g2, g3);
    *reinterpret_cast<uint2*>(g.next_a + static_cast<int64_t>(m) * g.d + col) =
        pack4_bf16(v.x * g0, v.y * g1, v.z * g2, v.w * g3);
    // the item's gpr consecutive lanes (gpr a power of two <= 32) sum their squares
    float sq = v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    const int lane = threadIdx.x & 31;
    const unsigned seg = gpr >= 32 ? 0xFFFFFFFFu : ((1u << gpr) - 1u) << (lane & ~(gpr - 1));
    for (int o = 1; o < gpr; o <<= 1) sq += __shfl_xor_sync(seg, sq, o);
    if ((lane & (gpr - 1)) == 0) atomicAdd(g.ss_out + m, sq);
}

// NB consecutive packed weight blocks (G_W_BYTES apart from wst) -> NB bf16 B
// buffers (G_B_BYTES apart from bst): this thread's RPP packed rows of column dq_n
// in each. A byte's two codes become the bf16 pair (128 + q_lo, 128 + q_hi) by a
// byte permute and a mask (exact), minus 136 gives q - 8 (exact), then
// (q - 8) s + (8 - z) s = (q - z) s in one bf16x2 fma. All loads of the NB blocks
// are issued before any arithmetic.
template <int NB>
__device__ __forceinline__ void dequant_blocks(const uint8_t* wst, uint8_t* bst, int dq_n, int dq_h) {
    constexpr int RPP = 32 / G_DQ_PARTS;
    static_assert(RPP == 16, "one 16-byte load of packed rows per block");
    uint32_t wl[NB][RPP / 4];
    __half sh[NB], zh[NB];
#pragma unroll
    for (int bb = 0; bb < NB; ++bb) {
        const uint8_t* wb = wst + bb * G_W_BYTES;
        const __half* sz = reinterpret_cast<const __half*>(wb + 32 * GT_N);
        sh[bb] = sz[dq_n];
        zh[bb] = sz[GT_N + dq_n];
        const uint4 v = *reinterpret_cast<const uint4*>(wb + dq_n * 32 + dq_h * RPP);
        wl[bb][0] = v.x;
        wl[bb][1] = v.y;
        wl[bb][2] = v.z;
        wl[bb][3] = v.w;
    }
    const __nv_bfloat162 k136 = __float2bfloat162_rn(136.0f);
#pragma unroll
    for (int bb = 0; bb < NB; ++bb) {
        const float sc = __half2float(sh[bb]);
        const __nv_bfloat162 s2 = __float2bfloat162_rn(sc);
        const __nv_bfloat162 zs2 = __float2bfloat162_rn((8.0f - __half2float(zh[bb])) * sc);
        uint32_t w[RPP];
#pragma unroll
        for (int wi = 0; wi < RPP / 4; ++wi) {
            const uint32_t lo = wl[bb][wi], hi = lo >> 4;
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const uint32_t x = (__byte_perm(lo, hi, b | ((4 + b) << 8)) & 0x000F000Fu) | 0x43004300u;
                __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&x);
                v = __hfma2(__hsub2(v, k136), s2, zs2);
                w[4 * wi + b] = *reinterpret_cast<const uint32_t*>(&v);
            }
        }
        uint8_t* row = bst + bb * G_B_BYTES + dq_n * 128;
#pragma unroll
        for (int q = 0; q < RPP / 4; ++q) {
            const int jj = dq_h * (RPP / 4) + q;
            *reinterpret_cast<uint4*>(row + ((jj ^ (dq_n & 7)) << 4)) =
                make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
        }
    }
}

// One 128-column tile over a 1/ks slice of the inputs; the ks CTAs of a tile are a
// cluster. Warp G_PROD_WARP streams each stage's packed weights (one bulk copy)
// into the weight ring and warp G_A_WARP its A tiles (one TMA box) into the A
// ring; the G_DQ_WARPS dequantising warps, in G_DQ_GROUPS groups that take
// alternate stages (one group's waits and latencies overlap the other's work),
// turn each stage's blocks into one of G_BP B stages (one wait and one arrival
// per stage, the two blocks' loads and arithmetic interleaved) and release the
// weight slot at once; warp G_MMA_WARP issues the MMAs and one commit per stage
// frees its A and B slots. The weights stream ahead of the dequantisation,
// bounded by it rather than by the MMAs. Then every CTA stages its fp32 partial
// tile in shared memory and, after a cluster barrier, finishes its share of the
// tile's columns from the ks partials (DSMEM reads).
template <int MODE>
__global__ void __launch_bounds__(G_THREADS, 1) w4_gemm_kernel(const __grid_constant__ GemmArgs g, void* ws) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* wfull = reinterpret_cast<uint64_t*>(smem + G_OFF_BAR);  // [G_WS]
    uint64_t* wempty = wfull + G_WS;                                    // [G_WS]
    uint64_t* afull = wempty + G_WS;                                    // [G_BP]
    uint64_t* bfull = afull + G_BP;                                     // [G_BP]
    uint64_t* cempty = bfull + G_BP;                                    // [G_BP]: A and B slots consumed
    uint64_t* acc_bar = cempty + G_BP;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_bar + 1);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t = blockIdx.x, sp = static_cast<int>(blockIdx.y) % g.ks;   // sp: the CTA's rank in its cluster
    const int kgi = static_cast<int>(blockIdx.y) / g.ks;                     // its K group
    const int n = item_count(g.n_max, g.n_dev);
    allow_dependents();   // the next kernel of the river may start launching
    if (n == 0) return;   // every CTA of the cluster leaves here
    const int kc = g.K / (g.ks * g.kg), k0 = (kgi * g.ks + sp) * kc, nkb = kc / GT_K;

    if (tid == 0) {
        for (int i = 0; i < G_WS; ++i) {
            tc::mbar_init(&wfull[i], 1);
            tc::mbar_init(&wempty[i], G_DQ_GWARPS);
        }
        for (int i = 0; i < G_BP; ++i) {
            tc::mbar_init(&afull[i], 1);
            tc::mbar_init(&bfull[i], G_DQ_GWARPS);
            tc::mbar_init(&cempty[i], 1);
        }
        tc::mbar_init(acc_bar, 1);
        *abort = 0;
        tc::fence_barrier_init();
    }
    if (warp == G_MMA_WARP) tc::tmem_alloc(tmem_slot, GT_N);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Launched early (programmatic dependent launch): the weights are constant, so
    // the producer streams the first stages' weights before it waits for the
    // previous kernel; everything else waits first.
    if (!(warp == G_PROD_WARP && lane == 0)) wait_prior_grid();
    if (g.ss_zero && t == 0 && blockIdx.y == 0)
        for (int i = tid; i < g.n_max; i += G_THREADS) g.ss_zero[i] = 0.f;

    const int nst = (nkb + G_BPS - 1) / G_BPS;
    // Stage j holds blocks 2 jr, 2 jr + 1 (jr = (j + rot) % nst): each tile walks its
    // stages from a different one (when all stages hold two blocks), so that the
    // tiles' CTAs, which all read the same A, ask for different A blocks at any
    // time; the MMAs only sum, in that order.
    const int rot = nkb % G_BPS == 0 ? t % nst : 0;

    if (warp == G_PROD_WARP) {
        // both packed weight blocks of stage j in one bulk copy into slot j % G_WS
        if (lane == 0) {
            const uint8_t* wsrc = g.blob + (static_cast<int64_t>(t) * (g.K / GT_K) + k0 / GT_K) * G_W_BYTES;
            int j = 0;
            for (; j < nst; ++j) {
                const int st = j % G_WS, jr = (j + rot) % nst;
                if (j >= G_WS && !tc::mbar_wait(&wempty[st], ((j / G_WS) - 1) & 1, abort, ws, 81)) break;
                const int nb = min(G_BPS, nkb - jr * G_BPS);
                tc::mbar_arrive_expect_tx(&wfull[st], nb * G_W_BYTES);
                bulk_load(smem + G_OFF_W + st * G_BPS * G_W_BYTES, wsrc + static_cast<int64_t>(jr) * G_BPS * G_W_BYTES,
                          nb * G_W_BYTES, &wfull[st]);
            }
            // stopped early: let the copies in flight land before the CTA moves on
            const uint64_t t0 = tc::globaltimer();
            for (int i = max(0, j - G_WS); i < j; ++i)
                while (!tc::mbar_test_wait(&wfull[i % G_WS], (i / G_WS) & 1) && tc::globaltimer() - t0 < 200000000ull) {
                }
        }
    } else if (warp == G_A_WARP) {
        // both A tiles of stage j in one TMA box (the k-blocks map) into slot j % G_BP
        if (lane == 0) {
            int j = 0;
            for (; j < nst; ++j) {
                const int sa = j % G_BP, jr = (j + rot) % nst;
                if (j >= G_BP && !tc::mbar_wait(&cempty[sa], ((j / G_BP) - 1) & 1, abort, ws, 87)) break;
                tc::mbar_arrive_expect_tx(&afull[sa], G_BPS * g.a_rows * GT_K * 2);
                tc::tma_load_3d(smem + G_OFF_A + sa * G_A_STAGE, &g.tm_a, 0, 0, k0 / GT_K + jr * G_BPS, &afull[sa]);
            }
            const uint64_t t0 = tc::globaltimer();
            for (int i = max(0, j - G_BP); i < j; ++i)
                while (!tc::mbar_test_wait(&afull[i % G_BP], (i / G_BP) & 1) && tc::globaltimer() - t0 < 200000000ull) {
                }
        }
    } else if (warp == G_MMA_WARP) {
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_bf16(GT_N, g.a_rows);   // M = columns, N = items
            for (int j = 0; j < nst; ++j) {
                const int bp = j % G_BP;
                if (!tc::mbar_wait(&afull[bp], (j / G_BP) & 1, abort, ws, 82)) break;
                if (!tc::mbar_wait(&bfull[bp], (j / G_BP) & 1, abort, ws, 83)) break;
                tc::tc_fence_after();
                for (int bb = 0; bb < G_BPS && j * G_BPS + bb < nkb; ++bb) {
                    const int kb = j * G_BPS + bb;
                    // the stage's blocks land a_rows x 128 bytes apart (one TMA box)
                    const uint64_t ad =
                        tc::smem_desc_sw128(tc::smem_u32(smem + G_OFF_A + bp * G_A_STAGE + bb * g.a_rows * 128));
                    const uint64_t bd = tc::smem_desc_sw128(tc::smem_u32(smem + G_OFF_B + (bp * G_BPS + bb) * G_B_BYTES));
#pragma unroll
                    for (int kk = 0; kk < GT_K / 16; ++kk)
                        tc::umma_bf16(tmem, bd + 2 * kk, ad + 2 * kk, idesc, kb | kk);
                }
                tc::umma_commit(&cempty[bp]);   // the stage's A and B slots
            }
            tc::umma_commit(acc_bar);   // every MMA issued has finished (also after a stop)
        }
    } else {
        // dequantiser: column dq_n, part dq_h of each k block (RPP packed rows, 2 RPP
        // inputs), both blocks of a stage per pass, the group's stages only
        const int gtid = tid % (G_DQ_GWARPS * 32);
        const int dq_n = gtid & 127, dq_h = gtid >> 7;
        for (int j = warp / G_DQ_GWARPS; j < nst; j += G_DQ_GROUPS) {
            const int st = j % G_WS, bp = j % G_BP;
            if (j >= G_BP && !tc::mbar_wait(&cempty[bp], ((j / G_BP) - 1) & 1, abort, ws, 84)) break;
            if (!tc::mbar_wait(&wfull[st], (j / G_WS) & 1, abort, ws, 85)) break;
            const uint8_t* wst = smem + G_OFF_W + st * G_BPS * G_W_BYTES;
            uint8_t* bst = smem + G_OFF_B + bp * G_BPS * G_B_BYTES;
            if (nkb - j * G_BPS >= 2)
                dequant_blocks<2>(wst, bst, dq_n, dq_h);
            else
                dequant_blocks<1>(wst, bst, dq_n, dq_h);
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
                tc::mbar_arrive(&wempty[st]);   // the packed codes have been read
                tc::mbar_arrive(&bfull[bp]);
            }
        }
    }
    // the accumulator is final
    if (warp < G_DQ_WARPS && !tc::mbar_wait(acc_bar, 0, abort, ws, 86)) *abort = 1;
    __syncthreads();
    const bool ok = !*abort;
    tc::tc_fence_after();
    // partial tile -> shared memory [item][column] (over the B ring, idle now): TMEM
    // lane = column, TMEM column = item; warp w reads lanes 32 (w % 4).. for items
    // 32 (w / 4).., lane l stores column 32 (w % 4) + l of each
    float* P = reinterpret_cast<float*>(smem + G_OFF_B);
    static_assert(G_DQ_WARPS / 4 * 32 == MAX_ITEMS, "the epilogue warps cover every item");
    if (ok && warp < G_DQ_WARPS) {
        const int c = (warp & 3) * 32 + lane;
        const int m0 = (warp >> 2) * 32;
        if (m0 < n) {   // warp-uniform
            float v[32];
            tc::tmem_ld32(tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + m0, v);
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (m0 + i < n) P[(m0 + i) * G_P_PITCH + c] = v[i];
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == G_MMA_WARP) tc::tmem_dealloc(tmem, GT_N);
    // every CTA of the cluster reaches both barriers (also after a stop)
    if (g.ks > 1) {
        cluster_arrive();
        cluster_wait();
    }
    if (ok && warp < G_DQ_WARPS) finish_tile<MODE>(g, P, t, n, sp);
    if (g.ks > 1) {   // no CTA leaves while a peer may still read its partial tile
        cluster_arrive();
        cluster_wait();
    }
}

// ------------------------------------------------------------------ attention
struct AttnArgs {
    CUtensorMap kmap, vmap;   // the caches, 5-D (head_dim, pos, head, seq, layer), box 64 x chunk, 128-byte swizzle
    int n_max;
    const int32_t* n_dev;
    int n_kv, qw;
    const bf16* qbuf;
    const int32_t* ipos;
    const int32_t* iseq;
    int layer;
    float qscale;          // log2(e) / sqrt(head_dim)
    bf16* obuf;            // [n][qw]
    void* ws;
    // the split-chunk kernel only
    int chunks;
    float* part;           // [n][n_kv][chunks][REP][HD + 2]
    int32_t* cnt;          // [n][n_kv]
};

// The pair walk (calls whose (item, kv head) pairs fill its consumer groups) is
// persistent: one CTA per SM, two consumer groups of four
// warps, each fed by its own producer warp through its own ring of AT_STAGES
// stages (a chunk of K and of V, TMA, one barrier each; the q rows, one bulk
// copy, with a pair's first chunk). A group takes every chunk of an (item, kv
// head) pair in order, so no chunk leaves a partial result: each warp keeps the
// online softmax (running maximum, sum and O) of its positions of every chunk in
// registers, and the four warps merge once, after the pair's last chunk. The
// pairs are ranked longest first (every CTA ranks the items the same way) and
// dealt to the groups in snake order, so that each group's chunks add up to
// about the same.
// In a chunk each warp takes WP positions: scores S^T = K Q^T (M = 16 positions,
// N = the kv head's query heads padded to 8, K = 16 columns of the head) and
// O^T += V^T P^T (M = 16 columns, N = the heads, K = 16 positions) as warp-level
// tensor-core products from registers, P^T coming from the score accumulators
// by an in-register transpose.
constexpr int AT_GROUPS = 2;                              // consumer groups
constexpr int AT_GT = 128;                                // threads of a group
constexpr int AT_PROD_WARP = AT_GROUPS * AT_GT / 32;      // warps 8 + g issue group g's copies
constexpr int AP_THREADS = (AT_PROD_WARP + AT_GROUPS) * 32;
constexpr int AT_STAGES = 3;
constexpr int AT_MAX_ITEMS = 128;

template <int HD, int REP>
struct AttnPairSmem {
    static constexpr int NW = AT_GT / 32;            // warps of a group
    static constexpr int CHUNK = at_pair_box(HD);    // positions per chunk
    static constexpr int WP = CHUNK / NW;            // positions per warp
    static constexpr int MT = WP / 16;               // 16-position tiles per warp
    static constexpr int KS = HD / 16;               // 16-column steps of a row
    static constexpr uint32_t KV_BYTES = CHUNK * HD * 2;     // 16 KB: halves of 64 columns, rows of 128 bytes
    static constexpr uint32_t STAGE = 2 * KV_BYTES + 2048;   // K | V | q rows (stages stay 1024-aligned)
    static constexpr uint32_t OFF_TAB = AT_GROUPS * AT_STAGES * STAGE;   // pos | seq | order, AT_MAX_ITEMS + 4 each
    static constexpr uint32_t OFF_BAR = OFF_TAB + 3 * (AT_MAX_ITEMS + 4) * 4;
    static constexpr size_t BYTES = 1024 + OFF_BAR + 3 * AT_GROUPS * AT_STAGES * 8 + 16;
    static_assert(REP <= 8 && MT >= 1 && WP % 16 == 0, "attention tiling");
    static_assert(REP * HD * 2 <= 2048, "q rows fit the stage");
    static_assert(NW * REP * HD * 4 <= KV_BYTES, "the warps' results fit the V buffer");
    static_assert(STAGE % 1024 == 0 && BYTES <= 232448, "shared memory");
};

// Byte offset of 16-byte piece q of row t in a swizzled K or V chunk: 64-column
// halves of CHUNK rows x 128 bytes, piece j of row t at j ^ (t % 8).
template <int CHUNK>
__device__ __forceinline__ uint32_t sw_off(int t, int q) {
    return (q >> 3) * (CHUNK * 128) + t * 128 + (((q & 7) ^ (t & 7)) << 4);
}

// Warp-level bf16 products with fp32 accumulation (16 x 8 x 16 per instruction;
// fragments as the PTX ISA's m16n8k16 layout: lane = 4 g + t holds rows g and
// g + 8, columns 2t and 2t + 1 of a C tile).
__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}
__device__ __forceinline__ void ldsm4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// bf16 pair, lo in the low half
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
// Barrier of consumer group grp (its 128 threads) that also returns whether v
// holds in every one of them. The aligned barrier wants each warp converged.
__device__ __forceinline__ bool group_all(int grp, bool v) {
    uint32_t r;
    __syncwarp();
    asm volatile(
        "{\n"
        ".reg .pred p, q;\n"
        "setp.ne.u32 p, %1, 0;\n"
        "bar.red.and.pred q, %2, %3, p;\n"
        "selp.u32 %0, 1, 0, q;\n"
        "}\n"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "r"(1 + grp), "r"(AT_GT)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void group_sync(int grp) {
    __syncwarp();
    asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "r"(AT_GT) : "memory");
}

// The k-th (item, kv head) pair of group gg (of G) in snake order over the
// ranked pairs, or -1 past the last.
__device__ __forceinline__ int snake_pair(int k, int gg, int G, int pairs) {
    const int p = k * G + ((k & 1) ? G - 1 - gg : gg);
    return p < pairs ? p : -1;
}

template <int HD, int REP>
__global__ void __launch_bounds__(AP_THREADS, 1) river_attn_pair_kernel(const __grid_constant__ AttnArgs a) {
    using S = AttnPairSmem<HD, REP>;
    constexpr int NW = S::NW, CHUNK = S::CHUNK, WP = S::WP, MT = S::MT, KS = S::KS;
    extern __shared__ uint8_t at_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(at_raw) + 1023) & ~uintptr_t(1023));
    int* s_pos = reinterpret_cast<int*>(sm + S::OFF_TAB);
    int* s_seq = s_pos + AT_MAX_ITEMS + 4;
    int* s_order = s_seq + AT_MAX_ITEMS + 4;   // the items, longest sequence first; then the skipped ones
    uint64_t* kfull = reinterpret_cast<uint64_t*>(sm + S::OFF_BAR);   // [group][stage]
    uint64_t* vfull = kfull + AT_GROUPS * AT_STAGES;
    uint64_t* empty = vfull + AT_GROUPS * AT_STAGES;
    volatile int* abort = reinterpret_cast<volatile int*>(empty + AT_GROUPS * AT_STAGES);
    __shared__ float s_mw[AT_GROUPS][NW][8], s_lw[AT_GROUPS][NW][8];   // the warps' maxima and sums per query head
    __shared__ int s_valid;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    allow_dependents();
    if (tid == 0) {
        for (int i = 0; i < AT_GROUPS * AT_STAGES; ++i) {
            tc::mbar_init(&kfull[i], 1);
            tc::mbar_init(&vfull[i], 1);
            tc::mbar_init(&empty[i], 1);
        }
        *abort = 0;
        tc::fence_barrier_init();
    }
    wait_prior_grid();   // q, the item table and the cache slots come from the q|k|v GEMM
    const int n = item_count(a.n_max, a.n_dev);
    for (int m = tid; m < n; m += AP_THREADS) {
        s_pos[m] = a.ipos[m];
        s_seq[m] = a.iseq[m];
    }
    __syncthreads();
    // rank the items by chunk count, longest first (ties by index; skipped items last)
    if (tid == 0) s_valid = 0;
    __syncthreads();
    for (int m = tid; m < n; m += AP_THREADS) {
        const int km = s_pos[m] >= 0 ? s_pos[m] / CHUNK + 1 : 0;
        int r = 0;
        for (int j = 0; j < n; ++j) {
            const int kj = s_pos[j] >= 0 ? s_pos[j] / CHUNK + 1 : 0;
            r += kj > km || (kj == km && j < m);
        }
        s_order[r] = m;
        if (km > 0) atomicAdd(&s_valid, 1);
    }
    __syncthreads();
    const int pairs = s_valid * a.n_kv;
    // a skipped item (position < 0) attends to nothing: its output rows are zero
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * AP_THREADS + tid; i < static_cast<int64_t>(n) * a.qw;
         i += static_cast<int64_t>(gridDim.x) * AP_THREADS) {
        const int m = static_cast<int>(i / a.qw);
        if (s_pos[m] < 0) a.obuf[i] = __float2bfloat16_rn(0.f);
    }
    const int G = AT_GROUPS * static_cast<int>(gridDim.x);

    if (warp >= AT_PROD_WARP) {   // group (warp - 8)'s copies
        const int grp = warp - AT_PROD_WARP, gg = static_cast<int>(blockIdx.x) * AT_GROUPS + grp;
        if (lane == 0) {
            uint64_t* kf = kfull + grp * AT_STAGES;
            uint64_t* vf = vfull + grp * AT_STAGES;
            uint64_t* em = empty + grp * AT_STAGES;
            int u = 0;   // chunks issued
            bool go = true;
            for (int k = 0; go; ++k) {
                const int p = snake_pair(k, gg, G, pairs);
                if (p < 0) break;
                const int m = s_order[p / a.n_kv], g = p % a.n_kv;
                const int nch = s_pos[m] / CHUNK + 1;
                for (int c = 0; c < nch; ++c, ++u) {
                    const int s = u % AT_STAGES;
                    if (*abort || (u >= AT_STAGES && !tc::mbar_wait(&em[s], ((u / AT_STAGES) - 1) & 1, abort, a.ws, 93))) {
                        go = false;
                        break;
                    }
                    uint8_t* st = sm + (grp * AT_STAGES + s) * S::STAGE;
                    const int t0 = c * CHUNK;
                    tc::mbar_arrive_expect_tx(&kf[s], S::KV_BYTES + (c == 0 ? REP * HD * 2 : 0));
#pragma unroll
                    for (int h = 0; h < HD / 64; ++h)
                        tc::tma_load_5d(st + h * (CHUNK * 128), &a.kmap, 64 * h, t0, g, s_seq[m], a.layer, &kf[s]);
                    if (c == 0)
                        bulk_load(st + 2 * S::KV_BYTES, a.qbuf + static_cast<int64_t>(m) * a.qw + g * REP * HD,
                                  REP * HD * 2, &kf[s]);
                    tc::mbar_arrive_expect_tx(&vf[s], S::KV_BYTES);
#pragma unroll
                    for (int h = 0; h < HD / 64; ++h)
                        tc::tma_load_5d(st + S::KV_BYTES + h * (CHUNK * 128), &a.vmap, 64 * h, t0, g, s_seq[m],
                                        a.layer, &vf[s]);
                }
            }
            // leave no copy in flight: wait (bounded, whether or not the block has
            // given up) for the last chunks issued to land
            const uint64_t t0 = tc::globaltimer();
            for (int j = u > AT_STAGES ? u - AT_STAGES : 0; j < u; ++j) {
                const uint32_t ph = (j / AT_STAGES) & 1;
                while (!(tc::mbar_test_wait(&kf[j % AT_STAGES], ph) && tc::mbar_test_wait(&vf[j % AT_STAGES], ph)) &&
                       tc::globaltimer() - t0 < 200000000ull) {
                }
            }
        }
        return;
    }

    // ---- consumer group grp: the chunks of its pairs, in the producer's order
    const int grp = warp / NW, gt = tid - grp * AT_GT, gw = gt >> 5;
    const int gg = static_cast<int>(blockIdx.x) * AT_GROUPS + grp;
    const int lg = lane >> 2, lt = lane & 3;    // fragment row group and column pair
    const int rr = lane & 7, mi = lane >> 3;    // lane l addresses row l % 8 of matrix l / 8 of an ldmatrix
    const int pw = gw * WP;                     // the warp's first position in a chunk
    const float qs = a.qscale;
    uint64_t* kf = kfull + grp * AT_STAGES;
    uint64_t* vf = vfull + grp * AT_STAGES;
    uint64_t* em = empty + grp * AT_STAGES;
    int u = 0;
    bool go = true;
    for (int k = 0; go; ++k) {
        const int p = snake_pair(k, gg, G, pairs);
        if (p < 0) break;
        const int m = s_order[p / a.n_kv], g = p % a.n_kv;
        const int pm = s_pos[m], nch = pm / CHUNK + 1;
        // this warp's running softmax over the pair's chunks (log2 domain): maximum
        // and this lane's share of the sum per query head 2t, 2t + 1, and O^T
        float mh[2] = {-INFINITY, -INFINITY}, lh[2] = {0.f, 0.f};
        float o[KS][4];
#pragma unroll
        for (int jj = 0; jj < KS; ++jj) o[jj][0] = o[jj][1] = o[jj][2] = o[jj][3] = 0.f;
        uint32_t qb[KS][2];
        for (int c = 0; c < nch; ++c, ++u) {
            const int s = u % AT_STAGES;
            const uint32_t ph = (u / AT_STAGES) & 1;
            if (!group_all(grp, tc::mbar_wait(&kf[s], ph, abort, a.ws, 95))) {
                go = false;
                break;
            }
            uint8_t* st = sm + (grp * AT_STAGES + s) * S::STAGE;
            uint8_t* s_v = st + S::KV_BYTES;
            if (c == 0) {   // Q^T fragments (heads past REP are zero), unscaled bf16
                const uint8_t* qrow = st + 2 * S::KV_BYTES + lg * HD * 2;
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
                    qb[kk][0] = lg < REP ? *reinterpret_cast<const uint32_t*>(qrow + (16 * kk + 2 * lt) * 2) : 0u;
                    qb[kk][1] = lg < REP ? *reinterpret_cast<const uint32_t*>(qrow + (16 * kk + 2 * lt + 8) * 2) : 0u;
                }
            }
            const int cnt = min(CHUNK, pm + 1 - c * CHUNK);
            uint32_t pb[MT][2];
            if (pw < cnt) {
                float sc[MT][4];
                const uint32_t kbase = tc::smem_u32(st);
#pragma unroll
                for (int i = 0; i < MT; ++i) {
                    sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
                    const int row = pw + 16 * i + ((mi & 1) << 3) + rr;   // a0 / a1: rows g, g + 8; a2 / a3: columns + 8
#pragma unroll
                    for (int kk = 0; kk < KS; ++kk) {
                        uint32_t fa[4];
                        ldsm4(kbase + sw_off<CHUNK>(row, 2 * kk + (mi >> 1)), fa);
                        mma16816(sc[i], fa, qb[kk][0], qb[kk][1]);
                    }
                }
                if (pw + WP > cnt) {   // the sequence ends inside this warp's positions
#pragma unroll
                    for (int i = 0; i < MT; ++i) {
                        const int p0 = pw + 16 * i + lg;
                        if (p0 >= cnt) sc[i][0] = sc[i][1] = -INFINITY;
                        if (p0 + 8 >= cnt) sc[i][2] = sc[i][3] = -INFINITY;
                    }
                }
                float cm[2] = {-INFINITY, -INFINITY};
#pragma unroll
                for (int i = 0; i < MT; ++i) {
                    cm[0] = fmaxf(cm[0], fmaxf(sc[i][0], sc[i][2]));
                    cm[1] = fmaxf(cm[1], fmaxf(sc[i][1], sc[i][3]));
                }
#pragma unroll
                for (int e = 0; e < 2; ++e) {
#pragma unroll
                    for (int sh = 4; sh < 32; sh <<= 1) cm[e] = fmaxf(cm[e], __shfl_xor_sync(0xFFFFFFFFu, cm[e], sh));
                    // to the log2 domain (s * log2(e) / sqrt(head_dim)); position pw is
                    // valid, so the new maximum is finite; the old one may be -inf
                    const float mn = fmaxf(mh[e], cm[e] * qs);
                    const float f = exp2f(mh[e] - mn);
                    lh[e] *= f;
#pragma unroll
                    for (int jj = 0; jj < KS; ++jj) {
                        o[jj][e] *= f;
                        o[jj][2 + e] *= f;
                    }
                    mh[e] = mn;
                }
#pragma unroll
                for (int i = 0; i < MT; ++i) {
                    const float p0 = exp2f(fmaf(sc[i][0], qs, -mh[0])), p1 = exp2f(fmaf(sc[i][1], qs, -mh[1]));
                    const float p2 = exp2f(fmaf(sc[i][2], qs, -mh[0])), p3 = exp2f(fmaf(sc[i][3], qs, -mh[1]));
                    lh[0] += p0 + p2;
                    lh[1] += p1 + p3;
                    pb[i][0] = movm_t(pack_bf16(p0, p1));   // P^T rows 2t, 2t + 1 of this tile, query head g
                    pb[i][1] = movm_t(pack_bf16(p2, p3));
                }
            }
            const bool vok = __all_sync(0xFFFFFFFFu, tc::mbar_wait(&vf[s], ph, abort, a.ws, 96));
            if (pw < cnt && vok) {
                if (pw + WP > cnt) {
                    // rows past the sequence hold whatever the cache slots hold (maybe
                    // not finite): zero them, since their weight 0 times a NaN would not vanish
                    constexpr int PR = (HD / 64) * 8;   // 16-byte pieces of a row
                    const int r0 = cnt - pw;
                    for (int idx = lane; idx < (WP - r0) * PR; idx += 32) {
                        const int row = pw + r0 + idx / PR, pc = idx % PR;
                        *reinterpret_cast<uint4*>(s_v + (pc >> 3) * (CHUNK * 128) + row * 128 + (pc & 7) * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_async_smem();   // before the next copies into this stage
                    __syncwarp();
                }
                const uint32_t vbase = tc::smem_u32(s_v);
#pragma unroll
                for (int jj = 0; jj < KS; ++jj)
#pragma unroll
                    for (int i = 0; i < MT; ++i) {
                        const int row = pw + 16 * i + ((mi >> 1) << 3) + rr;   // a0 / a2: positions 0-7 / 8-15 of the tile
                        uint32_t fa[4];
                        ldsm4_t(vbase + sw_off<CHUNK>(row, 2 * jj + (mi & 1)), fa);
                        mma16816(o[jj], fa, pb[i][0], pb[i][1]);
                    }
            }
            if (!group_all(grp, vok)) {   // every warp's reads of the stage are done
                go = false;
                break;
            }
            if (c == nch - 1) {
                // the pair's last chunk: merge the four warps' results by their
                // maxima, through this stage's V buffer
                float (*red)[REP][HD] = reinterpret_cast<float (*)[REP][HD]>(s_v);
#pragma unroll
                for (int e = 0; e < 2; ++e) {
#pragma unroll
                    for (int sh = 4; sh < 32; sh <<= 1) lh[e] += __shfl_xor_sync(0xFFFFFFFFu, lh[e], sh);
                    const int h = 2 * lt + e;
                    if (h < REP)
#pragma unroll
                        for (int jj = 0; jj < KS; ++jj) {   // O^T rows = columns 16 jj + g (+ 8)
                            red[gw][h][16 * jj + lg] = o[jj][e];
                            red[gw][h][16 * jj + lg + 8] = o[jj][2 + e];
                        }
                }
                if (lg == 0) {
                    s_mw[grp][gw][2 * lt] = mh[0];
                    s_mw[grp][gw][2 * lt + 1] = mh[1];
                    s_lw[grp][gw][2 * lt] = lh[0];
                    s_lw[grp][gw][2 * lt + 1] = lh[1];
                }
                fence_async_smem();   // before the next copies into this stage
                group_sync(grp);
                // warp 0 saw position 0, so M is finite; a warp that saw no position
                // has maximum -inf, weight 0 and O = 0
                bf16* out = a.obuf + static_cast<int64_t>(m) * a.qw + static_cast<int64_t>(g) * REP * HD;
                for (int i = gt; i < REP * HD; i += AT_GT) {
                    const int r = i / HD, e = i % HD;
                    float M = -INFINITY;
#pragma unroll
                    for (int w = 0; w < NW; ++w) M = fmaxf(M, s_mw[grp][w][r]);
                    float v = 0.f, L = 0.f;
#pragma unroll
                    for (int w = 0; w < NW; ++w) {
                        const float wt = exp2f(s_mw[grp][w][r] - M);
                        v = fmaf(red[w][r][e], wt, v);
                        L = fmaf(s_lw[grp][w][r], wt, L);
                    }
                    out[i] = __float2bfloat16_rn(v / L);
                }
                group_sync(grp);   // the merge's reads are done
            }
            if (gt == 0) tc::mbar_arrive(&em[s]);
        }
    }
}

template <int HD, int REP>
tee_status launch_attn_pair(const AttnArgs& a, cudaStream_t s) {
    static bool attr = false;
    constexpr size_t bytes = AttnPairSmem<HD, REP>::BYTES;
    if (!attr) {
        tee_status st = cuda_status(cudaFuncSetAttribute(river_attn_pair_kernel<HD, REP>,
                                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                         static_cast<int>(bytes)));
        if (st != TEE_OK) return st;
        attr = true;
    }
    const int64_t pairs = static_cast<int64_t>(a.n_max) * a.n_kv;
    const int grid = static_cast<int>(std::min<int64_t>(pairs, sm_count()));
    if (grid < 1) return TEE_OK;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(AP_THREADS);
    cfg.dynamicSmemBytes = bytes;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    tee_status st = cuda_status(cudaLaunchKernelEx(&cfg, river_attn_pair_kernel<HD, REP>, a));
    return st != TEE_OK ? st : launch_status();
}

// The split-chunk attention, for calls with fewer (item, kv head) pairs than
// the pair kernel has consumer groups (a pair walked by one group would leave
// most SMs idle): one CTA of four warps per (chunk of 256 / 128 positions, kv
// head, item), the same warp-level products as above on one chunk; a sequence
// of one chunk stores its output, otherwise the chunks' partials (o, m, l) go
// to the workspace and the last chunk to finish (a counter) merges them.
constexpr int AS_THREADS = 128;

template <int HD, int REP>
struct AttnSplitSmem {
    static constexpr int NW = AS_THREADS / 32;
    static constexpr int CHUNK = at_split_box(HD);   // positions per CTA
    static constexpr int WP = CHUNK / NW;            // positions per warp
    static constexpr int MT = WP / 16;               // 16-position tiles per warp
    static constexpr int KS = HD / 16;               // 16-column steps of a row
    static constexpr uint32_t KV_BYTES = CHUNK * HD * 2;   // 32 KB: halves of 64 columns, rows of 128 bytes
    static constexpr uint32_t OFF_K = 0;
    static constexpr uint32_t OFF_V = OFF_K + KV_BYTES;
    static constexpr uint32_t OFF_RED = OFF_V + KV_BYTES;
    static constexpr uint32_t OFF_BAR = OFF_RED + NW * REP * HD * 4;
    static constexpr size_t BYTES = 1024 + OFF_BAR + 64;
    static_assert(REP <= 8 && MT >= 1 && WP % 16 == 0, "attention tiling");
};

// One (chunk, kv head, item): TMA brings the chunk's K and V (swizzled) into
// shared memory. Each warp takes WP positions: scores S^T = K Q^T (M = 16
// positions, N = the kv head's query heads padded to 8, K = 16 columns of the
// head) and O^T += V^T P^T (M = 16 columns, N = the heads, K = 16 positions) as
// warp-level tensor-core products from registers; P^T comes from the score
// accumulators by an in-register transpose. The softmax of a warp's positions is
// taken on the accumulators; the warps' partial results are then merged by
// their maxima, and the last chunk of an (item, kv head) to finish merges the
// chunks' partials.
template <int HD, int REP>
__global__ void __launch_bounds__(AS_THREADS) river_attn_split_kernel(const __grid_constant__ AttnArgs a) {
    using S = AttnSplitSmem<HD, REP>;
    constexpr int NW = S::NW, CHUNK = S::CHUNK, WP = S::WP, MT = S::MT, KS = S::KS;
    extern __shared__ uint8_t at_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(at_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* s_v = sm + S::OFF_V;
    float (*s_red)[REP][HD] = reinterpret_cast<float (*)[REP][HD]>(sm + S::OFF_RED);
    uint64_t* kbar = reinterpret_cast<uint64_t*>(sm + S::OFF_BAR);
    uint64_t* vbar = kbar + 1;
    volatile int* abort = reinterpret_cast<volatile int*>(vbar + 1);
    __shared__ float s_mw[NW][8], s_lw[NW][8], s_ww[REP][NW];
    __shared__ float s_m[REP], s_sum[REP];
    __shared__ int s_last;

    const int c = blockIdx.x, g = blockIdx.y, m = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int lg = lane >> 2, lt = lane & 3;   // fragment row group and column pair
    allow_dependents();
    const int n = item_count(a.n_max, a.n_dev);
    if (m >= n) return;
    wait_prior_grid();   // q, the item table and the cache slots come from the q|k|v GEMM
    const int pm = a.ipos[m];
    bf16* out = a.obuf + static_cast<int64_t>(m) * a.qw + static_cast<int64_t>(g) * REP * HD;
    if (pm < 0) {   // a skipped item attends to nothing
        if (c == 0)
            for (int i = tid; i < REP * HD; i += AS_THREADS) out[i] = __float2bfloat16_rn(0.f);
        return;
    }
    const int nch = pm / CHUNK + 1;
    if (c >= nch) return;
    const int t0 = c * CHUNK, cnt = min(CHUNK, pm + 1 - t0);
    if (tid == 0) {
        tc::mbar_init(kbar, 1);
        tc::mbar_init(vbar, 1);
        *abort = 0;
        tc::fence_barrier_init();
        const uint32_t bytes = (HD / 64) * CHUNK * 128;
        const int sq = a.iseq[m];
        tc::mbar_arrive_expect_tx(kbar, bytes);
        for (int h = 0; h < HD / 64; ++h)
            tc::tma_load_5d(sm + S::OFF_K + h * (CHUNK * 128), &a.kmap, 64 * h, t0, g, sq, a.layer, kbar);
        tc::mbar_arrive_expect_tx(vbar, bytes);
        for (int h = 0; h < HD / 64; ++h)
            tc::tma_load_5d(s_v + h * (CHUNK * 128), &a.vmap, 64 * h, t0, g, sq, a.layer, vbar);
    }
    // Q^T fragments (columns 2t, 2t + 1 and 2t + 8, 2t + 9 of query head g; heads
    // past REP are zero), unscaled bf16: the softmax scale multiplies the fp32 scores
    uint32_t qb[KS][2];
    {
        const bf16* qrow = a.qbuf + static_cast<int64_t>(m) * a.qw + (static_cast<int64_t>(g) * REP + lg) * HD;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
            qb[kk][0] = lg < REP ? *reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 2 * lt) : 0u;
            qb[kk][1] = lg < REP ? *reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 2 * lt + 8) : 0u;
        }
    }
    __syncthreads();   // the barriers' initialisation
    const int pw = warp * WP;   // the warp's first position in the chunk
    const float qs = a.qscale;
    // lane l addresses row (l % 8) of matrix l / 8 of each ldmatrix; rows are 16-position tiles' rows
    const int rr = lane & 7, mi = lane >> 3;
    bool ok = tc::mbar_wait(kbar, 0, abort, a.ws, 91);
    float mh[2] = {-INFINITY, -INFINITY}, lh[2] = {0.f, 0.f};   // heads 2t and 2t + 1
    float o[KS][4];
#pragma unroll
    for (int j = 0; j < KS; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    uint32_t pb[MT][2];
    if (pw < cnt) {
        float s[MT][4];
        const uint32_t kbase = tc::smem_u32(sm + S::OFF_K);
#pragma unroll
        for (int i = 0; i < MT; ++i) {
            s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
            const int row = pw + 16 * i + ((mi & 1) << 3) + rr;   // a0 / a1: rows g, g + 8; a2 / a3: columns + 8
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
                uint32_t fa[4];
                ldsm4(kbase + sw_off<CHUNK>(row, 2 * kk + (mi >> 1)), fa);
                mma16816(s[i], fa, qb[kk][0], qb[kk][1]);
            }
        }
        if (pw + WP > cnt) {   // the sequence ends inside this warp's positions
#pragma unroll
            for (int i = 0; i < MT; ++i) {
                const int p0 = pw + 16 * i + lg;
                if (p0 >= cnt) s[i][0] = s[i][1] = -INFINITY;
                if (p0 + 8 >= cnt) s[i][2] = s[i][3] = -INFINITY;
            }
        }
#pragma unroll
        for (int i = 0; i < MT; ++i) {
            mh[0] = fmaxf(mh[0], fmaxf(s[i][0], s[i][2]));
            mh[1] = fmaxf(mh[1], fmaxf(s[i][1], s[i][3]));
        }
#pragma unroll
        for (int e = 0; e < 2; ++e)
#pragma unroll
            for (int sh = 4; sh < 32; sh <<= 1) mh[e] = fmaxf(mh[e], __shfl_xor_sync(0xFFFFFFFFu, mh[e], sh));
        // scores to the log2 domain: s * log2(e) / sqrt(head_dim); position pw is
        // valid, so the maxima are finite
        mh[0] *= qs;
        mh[1] *= qs;
#pragma unroll
        for (int i = 0; i < MT; ++i) {
            const float p0 = exp2f(fmaf(s[i][0], qs, -mh[0])), p1 = exp2f(fmaf(s[i][1], qs, -mh[1]));
            const float p2 = exp2f(fmaf(s[i][2], qs, -mh[0])), p3 = exp2f(fmaf(s[i][3], qs, -mh[1]));
            lh[0] += p0 + p2;
            lh[1] += p1 + p3;
            pb[i][0] = movm_t(pack_bf16(p0, p1));   // P^T rows 2t, 2t + 1 of this tile, query head g
            pb[i][1] = movm_t(pack_bf16(p2, p3));
        }
#pragma unroll
        for (int e = 0; e < 2; ++e)
#pragma unroll
            for (int sh = 4; sh < 32; sh <<= 1) lh[e] += __shfl_xor_sync(0xFFFFFFFFu, lh[e], sh);
    }
    ok = tc::mbar_wait(vbar, 0, abort, a.ws, 92) && ok;
    ok = __all_sync(0xFFFFFFFFu, ok);   // the warp-wide instructions below run in whole warps only
    if (pw < cnt && ok) {
        if (pw + WP > cnt) {
            // rows past the sequence hold whatever the cache slots hold (maybe not
            // finite): zero them, since their weight 0 times a NaN would not vanish
            constexpr int PR = (HD / 64) * 8;   // 16-byte pieces of a row
            const int r0 = cnt - pw;
            for (int idx = lane; idx < (WP - r0) * PR; idx += 32) {
                const int row = pw + r0 + idx / PR, pc = idx % PR;
                *reinterpret_cast<uint4*>(s_v + (pc >> 3) * (CHUNK * 128) + row * 128 + (pc & 7) * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
            __syncwarp();
        }
        const uint32_t vbase = tc::smem_u32(s_v);
#pragma unroll
        for (int j = 0; j < KS; ++j)
#pragma unroll
            for (int i = 0; i < MT; ++i) {
                const int row = pw + 16 * i + ((mi >> 1) << 3) + rr;   // a0 / a2: positions 0-7 / 8-15 of the tile
                uint32_t fa[4];
                ldsm4_t(vbase + sw_off<CHUNK>(row, 2 * j + (mi & 1)), fa);
                mma16816(o[j], fa, pb[i][0], pb[i][1]);
            }
        // O^T fragments: rows = columns 16 j + g (+ 8), columns = heads 2t, 2t + 1
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int h = 2 * lt + e;
            if (h < REP)
#pragma unroll
                for (int j = 0; j < KS; ++j) {
                    s_red[warp][h][16 * j + lg] = o[j][e];
                    s_red[warp][h][16 * j + lg + 8] = o[j][2 + e];
                }
        }
        if (lg == 0) {
            s_mw[warp][2 * lt] = mh[0];
            s_mw[warp][2 * lt + 1] = mh[1];
            s_lw[warp][2 * lt] = lh[0];
            s_lw[warp][2 * lt + 1] = lh[1];
        }
    }
    if (!ok) *abort = 1;
    __syncthreads();
    if (*abort) return;
    const int nwa = min(NW, (cnt + WP - 1) / WP);   // warps that saw positions
    if (tid < REP) {
        float M = -INFINITY;
        for (int w = 0; w < nwa; ++w) M = fmaxf(M, s_mw[w][tid]);
        float L = 0.f;
        for (int w = 0; w < nwa; ++w) {
            const float wt = exp2f(s_mw[w][tid] - M);
            s_ww[tid][w] = wt;
            L = fmaf(s_lw[w][tid], wt, L);
        }
        s_m[tid] = M;
        s_sum[tid] = L;
    }
    __syncthreads();
    if (nch == 1) {   // the whole range in this CTA: normalise and store
        for (int i = tid; i < REP * HD; i += AS_THREADS) {
            const int r = i / HD, e = i % HD;
            float v = 0.f;
            for (int w = 0; w < nwa; ++w) v = fmaf(s_red[w][r][e], s_ww[r][w], v);
            out[i] = __float2bfloat16_rn(v / s_sum[r]);
        }
        return;
    }
    float* pp = a.part + ((static_cast<int64_t>(m) * a.n_kv + g) * a.chunks + c) * (REP * (HD + 2));
    for (int i = tid; i < REP * HD; i += AS_THREADS) {
        const int r = i / HD, e = i % HD;
        float v = 0.f;
        for (int w = 0; w < nwa; ++w) v = fmaf(s_red[w][r][e], s_ww[r][w], v);
        pp[r * (HD + 2) + e] = v;
    }
    if (tid < REP) {
        pp[tid * (HD + 2) + HD] = s_m[tid];
        pp[tid * (HD + 2) + HD + 1] = s_sum[tid];
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        int32_t* ctr = a.cnt + m * a.n_kv + g;
        const int prev = atomicAdd(ctr, 1);
        s_last = prev == nch - 1;
        if (s_last) *ctr = 0;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // merge the chunks: O = sum_c o_c 2^(m_c - M) / sum_c l_c 2^(m_c - M). The
    // chunks' (m_c, l_c) go to shared memory first (one load per thread; the V
    // buffer is free by now), then a column's o_c are loaded 16 at a time.
    const int nc = a.chunks;
    const float* p0 = a.part + (static_cast<int64_t>(m) * a.n_kv + g) * nc * (REP * (HD + 2));
    float* s_ml = reinterpret_cast<float*>(s_v);   // [REP][nc][2] (the V chunk is no longer needed)
    float* s_w = s_ml + 2 * REP * nc;              // [REP][nc]: 2^(m_c - M) / L
    for (int i = tid; i < REP * nch; i += AS_THREADS) {
        const int r = i / nch, cc = i % nch;
        const float* q = p0 + cc * (REP * (HD + 2)) + r * (HD + 2) + HD;
        s_ml[(r * nc + cc) * 2] = __ldcg(q);
        s_ml[(r * nc + cc) * 2 + 1] = __ldcg(q + 1);
    }
    __syncthreads();
    if (tid < REP) {
        float M = -INFINITY;
        for (int cc = 0; cc < nch; ++cc) M = fmaxf(M, s_ml[(tid * nc + cc) * 2]);
        float L = 0.f;
        for (int cc = 0; cc < nch; ++cc) {
            const float w = exp2f(s_ml[(tid * nc + cc) * 2] - M);
            s_w[tid * nc + cc] = w;
            L = fmaf(s_ml[(tid * nc + cc) * 2 + 1], w, L);
        }
        for (int cc = 0; cc < nch; ++cc) s_w[tid * nc + cc] /= L;
    }
    __syncthreads();
    for (int i = tid; i < REP * HD; i += AS_THREADS) {
        const int r = i / HD, e = i % HD;
        float O = 0.f;
        for (int c0 = 0; c0 < nch; c0 += 16) {
            float v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (c0 + j < nch) v[j] = __ldcg(p0 + (c0 + j) * (REP * (HD + 2)) + r * (HD + 2) + e);
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (c0 + j < nch) O = fmaf(v[j], s_w[r * nc + c0 + j], O);
        }
        out[i] = __float2bfloat16_rn(O);
    }
}

template <int HD, int REP>
tee_status launch_attn_split(const AttnArgs& a, dim3 grid, cudaStream_t s) {
    static bool attr = false;
    constexpr size_t bytes = AttnSplitSmem<HD, REP>::BYTES;
    if (!attr) {
        tee_status st = cuda_status(cudaFuncSetAttribute(river_attn_split_kernel<HD, REP>,
                                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                         static_cast<int>(bytes)));
        if (st != TEE_OK) return st;
        attr = true;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(AS_THREADS);
    cfg.dynamicSmemBytes = bytes;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    tee_status st = cuda_status(cudaLaunchKernelEx(&cfg, river_attn_split_kernel<HD, REP>, a));
    return st != TEE_OK ? st : launch_status();
}

template <int HD, int REP>
tee_status launch_attn_rep(const AttnArgs& a, bool by_pair, cudaStream_t s) {
    return by_pair ? launch_attn_pair<HD, REP>(a, s) : launch_attn_split<HD, REP>(a, dim3(a.chunks, a.n_kv, a.n_max), s);
}

template <int HD>
tee_status launch_attn(const AttnArgs& a, int rep, bool by_pair, cudaStream_t s) {
    switch (rep) {
        case 1: return launch_attn_rep<HD, 1>(a, by_pair, s);
        case 2: return launch_attn_rep<HD, 2>(a, by_pair, s);
        case 4: return launch_attn_rep<HD, 4>(a, by_pair, s);
        case 8: return launch_attn_rep<HD, 8>(a, by_pair, s);
        default: return TEE_ERR_UNSUPPORTED;
    }
}

// ------------------------------------------------------------------ host
tee_status check_desc(const tee_river_desc* D) {
    if (!D) return TEE_ERR_INVALID_ARG;
    if (D->d <= 0 || D->n_q_heads <= 0 || D->n_kv_heads <= 0 || D->d_ff <= 0) return TEE_ERR_INVALID_ARG;
    if (D->flags != 0 && D->flags != TEE_RIVER_ATTN_BY_PAIR && D->flags != TEE_RIVER_ATTN_BY_CHUNK)
        return TEE_ERR_INVALID_ARG;
    if (!(D->eps >= 0.f) || !(D->rope_base > 0.f)) return TEE_ERR_INVALID_ARG;
    if (D->head_dim != 64 && D->head_dim != 128) return TEE_ERR_UNSUPPORTED;
    if (D->group != GT_K) return TEE_ERR_UNSUPPORTED;
    if (D->n_q_heads % D->n_kv_heads) return TEE_ERR_INVALID_ARG;
    const int rep = D->n_q_heads / D->n_kv_heads;
    if (rep != 1 && rep != 2 && rep != 4 && rep != 8) return TEE_ERR_UNSUPPORTED;
    const int qw = D->n_q_heads * D->head_dim, kvw = D->n_kv_heads * D->head_dim;
    if (D->d % GT_N || qw % GT_N || kvw % GT_N || D->d_ff % 64) return TEE_ERR_UNSUPPORTED;
    return TEE_OK;
}

bool seg_ok(const tee_w4& w) {
    return w.codes && w.scale && w.zero && aligned16(w.codes) && aligned16(w.scale) && aligned16(w.zero);
}

W4Seg seg_of(const tee_w4& w, int n) {
    return W4Seg{static_cast<const uint8_t*>(w.codes), static_cast<const __half*>(w.scale),
                 static_cast<const __half*>(w.zero), n};
}

// Packed weights of one exit layer: the q|k|v, o, gate|up and down GEMMs, each
// [tile][K / 64][G_W_BYTES] (a tile's k blocks contiguous, so that one bulk copy
// brings two of them).
struct LayerPack {
    size_t qkv, o, gu, dn, bytes;
};
LayerPack layer_pack(const tee_river_desc& D) {
    const size_t qw = static_cast<size_t>(D.n_q_heads) * D.head_dim, kvw = static_cast<size_t>(D.n_kv_heads) * D.head_dim;
    const size_t d = D.d, f = D.d_ff;
    auto sz = [](size_t tiles, size_t K) { return round_up(tiles * (K / GT_K) * G_W_BYTES, 256); };
    LayerPack p{};
    size_t o = 0;
    p.qkv = o;
    o += sz((qw + 2 * kvw) / GT_N, d);
    p.o = o;
    o += sz(d / GT_N, qw);
    p.gu = o;
    o += sz(f / 64, d);
    p.dn = o;
    o += sz(d / GT_N, f);
    p.bytes = o;
    return p;
}

// Repack the segments of one GEMM (q|k|v, o, gate|up interleaved per tile as 64 +
// 64 columns, down) into [tile][k block][codes | scales 128 | zeros 128], the codes
// of a block column by column ([128 columns][32 packed rows]: a column's 64 inputs
// in 32 consecutive bytes). Grid (tiles, K / 64), 128 threads: thread c fills column c.
__global__ void __launch_bounds__(128) w4_pack_kernel(W4Seg s0, W4Seg s1, W4Seg s2, int n_seg, int gu, int K,
                                                      uint8_t* __restrict__ blob) {
    const int t = blockIdx.x, kb = blockIdx.y, c = threadIdx.x;
    int si = 0, col;
    if (gu) {
        si = c >> 6;
        col = 64 * t + (c & 63);
    } else {
        int c0 = t * GT_N;
        const int n0 = s0.n, n1 = s1.n;
        if (n_seg > 1 && c0 >= n0) {
            c0 -= n0;
            si = 1;
            if (n_seg > 2 && c0 >= n1) {
                c0 -= n1;
                si = 2;
            }
        }
        col = c0 + c;
    }
    const W4Seg& sg = si == 0 ? s0 : (si == 1 ? s1 : s2);
    uint8_t* out = blob + (static_cast<int64_t>(t) * (K / GT_K) + kb) * G_W_BYTES;
    uint32_t word[8];
#pragma unroll
    for (int r = 0; r < 32; ++r) {
        const uint32_t b = sg.codes[static_cast<int64_t>(kb * 32 + r) * sg.n + col];
        if ((r & 3) == 0) word[r >> 2] = 0;
        word[r >> 2] |= b << (8 * (r & 3));
    }
    uint4* oc = reinterpret_cast<uint4*>(out + c * 32);
    oc[0] = make_uint4(word[0], word[1], word[2], word[3]);
    oc[1] = make_uint4(word[4], word[5], word[6], word[7]);
    __half* o16 = reinterpret_cast<__half*>(out + 32 * GT_N);
    o16[c] = sg.scale[static_cast<int64_t>(kb) * sg.n + col];
    o16[GT_N + c] = sg.zero[static_cast<int64_t>(kb) * sg.n + col];
}

tee_status pack_gemm(const W4Seg* segs, int n_seg, bool gu, int K, int tiles, uint8_t* blob, cudaStream_t s) {
    const W4Seg none = segs[0];
    w4_pack_kernel<<<dim3(tiles, K / GT_K), 128, 0, s>>>(segs[0], n_seg > 1 ? segs[1] : none,
                                                       n_seg > 2 ? segs[2] : none, n_seg, gu ? 1 : 0, K, blob);
    return launch_status();
}

// Clusters of ks GEMM CTAs that can be resident at once (one CTA per SM).
int max_clusters(int ks) {
    static int cache[MAX_KS + 1] = {};
    if (ks <= 1) return 1 << 20;
    if (cache[ks]) return cache[ks];
    if (cudaFuncSetAttribute(w4_gemm_kernel<M_O>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(G_SMEM)) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(1, ks * 64);
    cfg.blockDim = dim3(G_THREADS);
    cfg.dynamicSmemBytes = G_SMEM;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = ks;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int c = 0;
    if (cudaOccupancyMaxActiveClusters(&c, w4_gemm_kernel<M_O>, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        c = 0;
    }
    cache[ks] = c > 0 ? c : -1;
    return c;
}

template <int MODE>
tee_status launch_gemm(const GemmArgs& g0, void* ws, cudaStream_t s) {
    GemmArgs g = g0;
    g.a_rows = std::min(G_A_ROWS, (g.n_max + 15) / 16 * 16);   // the MMA's N: a multiple of 16
    tee_status st = make_tmap_bf16_kblocks(&g.tm_a, g.a, G_A_ROWS, static_cast<uint64_t>(g.lda) * 2, g.K / GT_K,
                                           g.a_rows, G_BPS);
    if (st != TEE_OK) return st;
    static bool attr = false;
    if (!attr) {
        st = cuda_status(cudaFuncSetAttribute(w4_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              static_cast<int>(G_SMEM)));
        if (st != TEE_OK) return st;
        attr = true;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(g.N / GT_N, g.ks * g.kg);
    cfg.blockDim = dim3(G_THREADS);
    cfg.dynamicSmemBytes = G_SMEM;
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    at[1].id = cudaLaunchAttributeClusterDimension;
    at[1].val.clusterDim.x = 1;
    at[1].val.clusterDim.y = g.ks;
    at[1].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = g.ks > 1 ? 2 : 1;
    st = cuda_status(cudaLaunchKernelEx(&cfg, w4_gemm_kernel<MODE>, g, ws));
    return st != TEE_OK ? st : launch_status();
}

}  // namespace

}  // namespace tee

using namespace tee;

extern "C" size_t tee_exit_river_prep_size(const tee_river_desc* D, int32_t n_layers, int32_t max_pos) {
    if (check_desc(D) != TEE_OK || max_pos <= 0 || n_layers < 0) return 0;
    return PREP_HEADER_BYTES + static_cast<size_t>(n_layers) * layer_pack(*D).bytes +
           rope_table_bytes(max_pos, D->head_dim);
}

extern "C" tee_status tee_exit_river_prepare(const tee_river_desc* D, int32_t n_layers, const tee_river_layer* layers,
                                             int32_t max_pos, void* prep, size_t prep_bytes, void* stream) {
    tee_status st = check_desc(D);
    if (st != TEE_OK) return st;
    if (max_pos <= 0 || n_layers < 0 || (n_layers > 0 && !layers)) return TEE_ERR_INVALID_ARG;
    if (!prep || !aligned16(prep) || prep_bytes < tee_exit_river_prep_size(D, n_layers, max_pos))
        return TEE_ERR_WORKSPACE;
    for (int l = 0; l < n_layers; ++l) {
        const tee_river_layer& L = layers[l];
        if (!seg_ok(L.wq) || !seg_ok(L.wk) || !seg_ok(L.wv) || !seg_ok(L.wo) || !seg_ok(L.wg) || !seg_ok(L.wu) ||
            !seg_ok(L.wd))
            return TEE_ERR_INVALID_ARG;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    PrepHeader h{};
    h.magic = RIVER_MAGIC;
    h.d = D->d;
    h.n_kv_heads = D->n_kv_heads;
    h.head_dim = D->head_dim;
    h.max_pos = max_pos;
    h.n_layers = n_layers;
    st = cuda_status(cudaMemcpyAsync(prep, &h, sizeof(h), cudaMemcpyHostToDevice, s));
    if (st != TEE_OK) return st;
    const int d = D->d, qw = D->n_q_heads * D->head_dim, kvw = D->n_kv_heads * D->head_dim, f = D->d_ff;
    const LayerPack lp = layer_pack(*D);
    for (int l = 0; l < n_layers; ++l) {
        const tee_river_layer& L = layers[l];
        uint8_t* base = static_cast<uint8_t*>(prep) + PREP_HEADER_BYTES + l * lp.bytes;
        const W4Seg qkv[3] = {seg_of(L.wq, qw), seg_of(L.wk, kvw), seg_of(L.wv, kvw)};
        const W4Seg o[1] = {seg_of(L.wo, d)};
        const W4Seg gu[2] = {seg_of(L.wg, f), seg_of(L.wu, f)};
        const W4Seg dn[1] = {seg_of(L.wd, d)};
        if ((st = pack_gemm(qkv, 3, false, d, (qw + 2 * kvw) / GT_N, base + lp.qkv, s)) != TEE_OK) return st;
        if ((st = pack_gemm(o, 1, false, qw, d / GT_N, base + lp.o, s)) != TEE_OK) return st;
        if ((st = pack_gemm(gu, 2, true, d, f / 64, base + lp.gu, s)) != TEE_OK) return st;
        if ((st = pack_gemm(dn, 1, false, f, d / GT_N, base + lp.dn, s)) != TEE_OK) return st;
    }
    float2* table = reinterpret_cast<float2*>(static_cast<char*>(prep) + PREP_HEADER_BYTES + n_layers * lp.bytes);
    return build_rope_table(table, max_pos, D->head_dim / 2, D->rope_base, s);
}

extern "C" size_t tee_exit_river_workspace_size(const tee_river_desc* D, int32_t n_max, int32_t max_pos) {
    if (check_desc(D) != TEE_OK || n_max < 0 || n_max > MAX_ITEMS || max_pos <= 0) return 0;
    return river_ws(*D, n_max, max_pos).end;
}

extern "C" tee_status tee_exit_river(const tee_river_desc* D, int32_t n_layers, const tee_river_layer* layers,
                                     const void* prep, size_t prep_bytes, int32_t n_max, const int32_t* n_dev,
                                     const void* h, int64_t ld_h, int32_t h_rows, const int32_t* rows,
                                     const int32_t* pos, const int32_t* seq, void* k_cache, void* v_cache,
                                     const tee_cache_layout* cache, void* h_out, int64_t ld_out, void* ws,
                                     size_t ws_bytes, void* stream) {
    tee_status st = check_desc(D);
    if (st != TEE_OK) return st;
    if (n_layers < 0 || n_max < 0 || n_max > MAX_ITEMS || (n_layers > 0 && !layers) || !cache) return TEE_ERR_INVALID_ARG;
    if (n_layers == 0 || n_max == 0) return TEE_OK;
    if (!h || !pos || !k_cache || !v_cache || !h_out || h_rows < 0) return TEE_ERR_INVALID_ARG;
    if (!aligned16(h) || !aligned16(h_out) || (ld_h * 2) % 16 || (ld_out * 2) % 16 || ld_h < D->d || ld_out < D->d)
        return TEE_ERR_INVALID_ARG;
    const int d = D->d, hd = D->head_dim, qw = D->n_q_heads * hd, kvw = D->n_kv_heads * hd, f = D->d_ff;
    const tee_cache_layout& cl = *cache;
    if (cl.n_heads < D->n_kv_heads || cl.max_pos <= 0 || cl.n_seq <= 0 || cl.n_layers <= 0) return TEE_ERR_INVALID_ARG;
    if (!aligned16(k_cache) || !aligned16(v_cache) || cl.s_layer % 8 || cl.s_seq % 8 || cl.s_head % 8 || cl.s_pos % 8)
        return TEE_ERR_INVALID_ARG;
    for (int l = 0; l < n_layers; ++l) {
        const tee_river_layer& L = layers[l];
        if (!L.attn_norm || !L.ffn_norm || !aligned16(L.attn_norm) || !aligned16(L.ffn_norm)) return TEE_ERR_INVALID_ARG;
        if (L.cache_layer < 0 || L.cache_layer >= cl.n_layers) return TEE_ERR_INVALID_ARG;
    }
    const LayerPack lp = layer_pack(*D);
    if (!prep || !aligned16(prep) || prep_bytes < tee_exit_river_prep_size(D, n_layers, 1)) return TEE_ERR_WORKSPACE;
    const RiverWs w = river_ws(*D, n_max, cl.max_pos);
    if (!ws || ws_bytes < w.end) return TEE_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const PrepHeader* hdr = static_cast<const PrepHeader*>(prep);
    const float2* rope =
        reinterpret_cast<const float2*>(static_cast<const char*>(prep) + PREP_HEADER_BYTES + n_layers * lp.bytes);

    float* resid = ws_at<float>(ws, w.resid);
    bf16* abuf = ws_at<bf16>(ws, w.abuf);
    bf16* qbuf = ws_at<bf16>(ws, w.qbuf);
    bf16* obuf = ws_at<bf16>(ws, w.obuf);
    bf16* act = ws_at<bf16>(ws, w.act);
    float* ss_a = ws_at<float>(ws, w.ss_a);
    float* ss_f = ws_at<float>(ws, w.ss_f);
    int32_t* ipos = ws_at<int32_t>(ws, w.ipos);
    int32_t* iseq = ws_at<int32_t>(ws, w.iseq);
    int32_t* acnt = ws_at<int32_t>(ws, w.acnt);

    GatherArgs ga{};
    ga.n_max = n_max;
    ga.n_dev = n_dev;
    ga.h = static_cast<const bf16*>(h);
    ga.ld_h = ld_h;
    ga.h_rows = h_rows;
    ga.rows = rows;
    ga.pos = pos;
    ga.seq = seq;
    ga.cl = cl;
    ga.hdr = hdr;
    ga.d = d;
    ga.gain = static_cast<const bf16*>(layers[0].attn_norm);
    ga.resid = resid;
    ga.abuf = abuf;
    ga.ss_a = ss_a;
    ga.ss_f = ss_f;
    ga.ipos = ipos;
    ga.iseq = iseq;
    ga.cnt = acnt;
    ga.n_cnt = KG_CNT + (w.by_pair ? 0 : n_max * D->n_kv_heads);
    river_gather_kernel<<<n_max, 256, 0, s>>>(ga, ws);
    if ((st = launch_status()) != TEE_OK) return st;

    GemmArgs g{};
    g.kg_cnt = acnt;   // cleared by the prologue
    g.n_max = n_max;
    g.n_dev = n_dev;
    g.eps = D->eps;
    g.qw = qw;
    g.kvw = kvw;
    g.hd = hd;
    g.half = hd / 2;
    g.qbuf = qbuf;
    g.ipos = ipos;
    g.iseq = iseq;
    g.rope = rope;
    g.kc = static_cast<bf16*>(k_cache);
    g.vc = static_cast<bf16*>(v_cache);
    g.cl = cl;
    g.resid = resid;
    g.d = d;
    g.act = act;
    g.d_ff = f;
    g.ld_out = ld_out;

    AttnArgs at{};
    at.n_max = n_max;
    at.n_dev = n_dev;
    at.n_kv = D->n_kv_heads;
    at.qw = qw;
    at.qbuf = qbuf;
    at.ipos = ipos;
    at.iseq = iseq;
    const int box = w.by_pair ? at_pair_box(hd) : at_split_box(hd);
    if ((st = make_tmap_cache(&at.kmap, k_cache, hd, cl, box)) != TEE_OK) return st;
    if ((st = make_tmap_cache(&at.vmap, v_cache, hd, cl, box)) != TEE_OK) return st;
    at.qscale = 1.4426950408889634f / sqrtf(static_cast<float>(hd));
    at.obuf = obuf;
    at.ws = ws;
    const int rep = D->n_q_heads / D->n_kv_heads;
    if (!w.by_pair) {
        at.chunks = attn_chunks(*D, cl.max_pos);
        at.part = ws_at<float>(ws, w.apart);
        at.cnt = acnt + KG_CNT;
        if (!split_merge_fits(*D, cl.max_pos)) return TEE_ERR_UNSUPPORTED;   // the chunk walk forced
    }

    for (int l = 0; l < n_layers; ++l) {
        const tee_river_layer& L = layers[l];
        const bool last = l == n_layers - 1;
        // q | k | v
        const uint8_t* lbase = static_cast<const uint8_t*>(prep) + PREP_HEADER_BYTES + l * lp.bytes;
        g.blob = lbase + lp.qkv;
        g.K = d;
        g.N = qw + 2 * kvw;
        g.ks = choose_ks(g.N / GT_N, d);
        g.kg = 1;
        g.a = abuf;
        g.lda = d;
        g.ss_in = ss_a;
        g.inv_width = 1.0f / d;
        g.ss_zero = nullptr;
        g.layer = L.cache_layer;
        if ((st = launch_gemm<M_QKV>(g, ws, s)) != TEE_OK) return st;
        // attention
        at.layer = L.cache_layer;
        st = hd == 64 ? launch_attn<64>(at, rep, w.by_pair, s) : launch_attn<128>(at, rep, w.by_pair, s);
        if (st != TEE_OK) return st;
        // h1 = h + o Wo
        g.blob = lbase + lp.o;
        g.K = qw;
        g.N = d;
        g.ks = choose_ks(d / GT_N, qw);
        g.kg = choose_kg(d / GT_N, g.ks, qw);
        g.a = obuf;
        g.lda = qw;
        g.ss_in = nullptr;
        g.next_gain = static_cast<const bf16*>(L.ffn_norm);
        g.next_a = abuf;
        g.ss_out = ss_f;
        g.h_out = nullptr;
        if ((st = launch_gemm<M_O>(g, ws, s)) != TEE_OK) return st;
        // a = SiLU(x2 Wg) * (x2 Wu)
        g.blob = lbase + lp.gu;
        g.K = d;
        g.N = 2 * f;
        g.ks = choose_ks(g.N / GT_N, d);
        g.kg = 1;
        g.a = abuf;
        g.lda = d;
        g.ss_in = ss_f;
        g.ss_zero = ss_a;
        if ((st = launch_gemm<M_GU>(g, ws, s)) != TEE_OK) return st;
        // h2 = h1 + a Wd
        g.blob = lbase + lp.dn;
        g.K = f;
        g.N = d;
        g.ks = choose_ks(d / GT_N, f);
        g.kg = choose_kg(d / GT_N, g.ks, f);
        g.a = act;
        g.lda = f;
        g.ss_in = nullptr;
        g.ss_zero = ss_f;
        if (last) {
            g.h_out = static_cast<bf16*>(h_out);
            g.next_gain = nullptr;
            g.next_a = nullptr;
            g.ss_out = nullptr;
        } else {
            g.h_out = nullptr;
            g.next_gain = static_cast<const bf16*>(layers[l + 1].attn_norm);
            g.next_a = abuf;
            g.ss_out = ss_a;
        }
        if ((st = launch_gemm<M_DOWN>(g, ws, s)) != TEE_OK) return st;
    }
    return TEE_OK;
}
