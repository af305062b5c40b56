// The Exit River (River-LLM, core method and method steps 1 and 3): the tokens
// that left the backbone run the W4A16 copies of the remaining decoder layers,
// each of which writes the skipped layer's K/V into the backbone's slots.
//
// One call = a prologue kernel and, per exit layer, five launches:
//   river_gather        h rows -> fp32 residual stream, bf16 (h * attn_norm),
//                       sum(h^2) per item; item checks; counters cleared
//   w4_gemm<QKV>        [q|k|v] = (h * g) . [Wq|Wk|Wv], times 1/rms(h); RoPE on
//                       q and k; q to the workspace, k and v to the cache slot
//   river_attn          per (item, kv head, chunk of 256 / 128 positions):
//                       scores, partial softmax and P.V on the CUDA cores (a
//                       bandwidth-bound read of the cache); the last chunk of an
//                       (item, kv head) merges the partials
//   w4_gemm<O>          h1 = h + o . Wo; bf16 (h1 * ffn_norm) and sum(h1^2)
//   w4_gemm<GU>         gate | up from (h1 * g2) . [Wg|Wu] (64 columns of each
//                       per tile), times 1/rms(h1); a = SiLU(gate) * up (bf16)
//   w4_gemm<DOWN>       h2 = h1 + a . Wd; bf16 (h2 * next attn_norm) and
//                       sum(h2^2), or h_out = bf16(h2) after the last layer
// RMSNorm's row scale commutes out of the contraction: A holds h * g in bf16
// and the epilogue multiplies by 1/rms, whose sum of squares the producing
// kernel accumulated in fp32.
//
// w4_gemm (tcgen05): a CTA computes a 128-column tile for every item (M = 128
// TMEM lanes, items <= 128) over a 1/ks slice of the inputs. cp.async brings
// the int4 codes (a deep ring: the weights are the DRAM traffic), the fp16
// scales/zeros and the bf16 A tile (128-byte swizzle); every thread then
// dequantises 32 weights of the 128 x 64 B tile into shared memory, and one
// thread issues four 128x128x16 MMAs into TMEM. Split-K partials go to the
// workspace; the CTA that finishes a tile last (an arrival counter) sums them
// in split order and runs the epilogue.
#include <algorithm>

#include "fill.cuh"
#include "tc.cuh"

namespace tee {

namespace {

using bf16 = __nv_bfloat16;

constexpr uint32_t RIVER_MAGIC = 0x54455256u;  // "TERV"

// ------------------------------------------------------------------ workspace
struct RiverWs {
    size_t resid, abuf, qbuf, obuf, act, ss_a, ss_f, ipos, iseq, gcnt, acnt, part, apart, end;
};

constexpr int GT_N = 128;        // output columns per GEMM tile
constexpr int GT_K = 64;         // inputs per k block
constexpr int G_THREADS = 256;
constexpr int G_CS = 8;          // code / scale ring depth (blocks)
constexpr int G_AS = 4;          // A ring depth
constexpr uint32_t G_A_BYTES = 128 * GT_K * 2;       // 16 KB: 128 rows x 64 bf16
constexpr uint32_t G_B_BYTES = GT_N * GT_K * 2;      // 16 KB
constexpr uint32_t G_C_BYTES = 32 * GT_N;            // 4 KB: 32 packed rows x 128 columns
constexpr uint32_t G_SZ_BYTES = 2 * GT_N * 2;        // 512 B: scales, zeros
constexpr uint32_t G_OFF_A = 0;
constexpr uint32_t G_OFF_B = G_OFF_A + G_AS * G_A_BYTES;
constexpr uint32_t G_OFF_C = G_OFF_B + 2 * G_B_BYTES;
constexpr uint32_t G_OFF_SZ = G_OFF_C + G_CS * G_C_BYTES;
constexpr uint32_t G_OFF_BAR = G_OFF_SZ + G_CS * G_SZ_BYTES;
constexpr size_t G_SMEM = 1024 + G_OFF_BAR + 64;
static_assert(G_OFF_B % 1024 == 0 && G_OFF_C % 16 == 0 && G_OFF_BAR % 8 == 0, "alignment");

constexpr int MAX_KS = 16;
constexpr int MAX_ITEMS = 128;

int max_tiles(const tee_river_desc& D) {
    const int qkv = (D.n_q_heads + 2 * D.n_kv_heads) * D.head_dim / GT_N;
    const int gu = D.d_ff / 64;
    const int dd = D.d / GT_N;
    return std::max(qkv, std::max(gu, dd));
}

int at_chunk(int hd) { return hd == 64 ? 256 : 128; }

// K splits: the largest power of two that keeps tiles * ks within the SMs and
// leaves each split at least two 64-input blocks.
int choose_ks(int tiles, int K) {
    const int sms = sm_count();
    int ks = 1;
    while (ks * 2 <= MAX_KS && tiles * ks * 2 <= sms && K % (ks * 2 * GT_K) == 0 && K / (ks * 2) >= 2 * GT_K)
        ks *= 2;
    return ks;
}

// Largest ks * N of the layer's four GEMMs (the split-K partials).
size_t part_cols(const tee_river_desc& D) {
    const size_t qw = static_cast<size_t>(D.n_q_heads) * D.head_dim, kvw = static_cast<size_t>(D.n_kv_heads) * D.head_dim;
    const size_t nq = qw + 2 * kvw, nf = 2 * static_cast<size_t>(D.d_ff);
    size_t m = nq * choose_ks(static_cast<int>(nq / GT_N), D.d);
    m = std::max(m, static_cast<size_t>(D.d) * choose_ks(D.d / GT_N, static_cast<int>(qw)));
    m = std::max(m, nf * choose_ks(static_cast<int>(nf / GT_N), D.d));
    m = std::max(m, static_cast<size_t>(D.d) * choose_ks(D.d / GT_N, D.d_ff));
    return m;
}

RiverWs river_ws(const tee_river_desc& D, int n_max, int max_pos) {
    const size_t n = static_cast<size_t>(n_max > 0 ? n_max : 1);
    const size_t d = D.d, qw = static_cast<size_t>(D.n_q_heads) * D.head_dim, f = D.d_ff;
    const int rep = D.n_q_heads / std::max(1, D.n_kv_heads);
    const size_t chunks = (static_cast<size_t>(max_pos) + at_chunk(D.head_dim) - 1) / at_chunk(D.head_dim);
    RiverWs w{};
    size_t o = TEE_WS_HEADER_BYTES;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = round_up(o + bytes, 256);
        return at;
    };
    w.resid = take(n * d * 4);
    w.abuf = take(n * d * 2);
    w.qbuf = take(n * qw * 2);
    w.obuf = take(n * qw * 2);
    w.act = take(n * f * 2);
    w.ss_a = take(n * 4);
    w.ss_f = take(n * 4);
    w.ipos = take(n * 4);
    w.iseq = take(n * 4);
    w.gcnt = take(static_cast<size_t>(max_tiles(D)) * 4);
    w.acnt = take(n * D.n_kv_heads * 4);
    w.part = take(n * part_cols(D) * 4);
    w.apart = take(n * D.n_kv_heads * chunks * rep * (D.head_dim + 2) * 4);
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
    int32_t* cnt;   // GEMM tile counters then attention counters
    int n_cnt;
};

__global__ void __launch_bounds__(256) river_gather_kernel(GatherArgs a, void* ws) {
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
    W4Seg seg[3];
    int n_seg, K, N, ks;
    int n_max;
    const int32_t* n_dev;
    const bf16* a;          // [n][lda]
    int64_t lda;
    float* part;            // [ks][n_max][N]
    int32_t* cnt;           // [tiles]
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

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(tc::smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Column c (0..127) of tile t -> (segment, column within it).
template <int MODE>
__device__ __forceinline__ void tile_col(const GemmArgs& g, int t, int c, int& s, int& col) {
    if (MODE == M_GU) {
        s = c >> 6;
        col = 64 * t + (c & 63);
    } else {
        int c0 = t * GT_N;
        s = 0;
        while (s + 1 < g.n_seg && c0 >= g.seg[s].n) {
            c0 -= g.seg[s].n;
            ++s;
        }
        col = c0 + c;
    }
}

__device__ __forceinline__ float row_scale(const GemmArgs& g, int m) {
    return g.ss_in ? 1.0f / sqrtf(g.ss_in[m] * g.inv_width + g.eps) : 1.f;
}

// Split-K partial sum of (item m, tile column c), in split order.
__device__ __forceinline__ float part_sum(const GemmArgs& g, int m, int col) {
    float v = 0.f;
    for (int s = 0; s < g.ks; ++s) v += __ldcg(g.part + (static_cast<int64_t>(s) * g.n_max + m) * g.N + col);
    return v;
}

template <int MODE>
__device__ void finish_tile(const GemmArgs& g, int t, int n, void* ws) {
    const int tid = threadIdx.x;
    const int c0 = t * GT_N;
    if (MODE == M_QKV) {
        const int pairs = GT_N / 2;
        for (int idx = tid; idx < n * pairs; idx += G_THREADS) {
            const int m = idx / pairs, p = idx % pairs;
            const int ht = p / g.half, i = p % g.half;
            const int lo = c0 + ht * g.hd + i, hi = lo + g.half;
            const int pm = g.ipos[m];
            if (pm < 0) continue;
            const float rs = row_scale(g, m);
            float x1 = part_sum(g, m, lo) * rs, x2 = part_sum(g, m, hi) * rs;
            const bool is_v = lo >= g.qw + g.kvw;
            if (!is_v) {
                const float2 cs = g.rope[static_cast<int64_t>(pm) * g.half + i];
                const float y1 = x1 * cs.x - x2 * cs.y, y2 = x2 * cs.x + x1 * cs.y;
                x1 = y1;
                x2 = y2;
            }
            if (lo < g.qw) {
                bf16* q = g.qbuf + static_cast<int64_t>(m) * g.qw;
                q[lo] = __float2bfloat16_rn(x1);
                q[hi] = __float2bfloat16_rn(x2);
            } else {
                const int cc = is_v ? lo - g.qw - g.kvw : lo - g.qw;
                const int head = cc / g.hd, e = cc % g.hd;
                bf16* dst = (is_v ? g.vc : g.kc) + g.layer * g.cl.s_layer + g.iseq[m] * g.cl.s_seq +
                            head * g.cl.s_head + static_cast<int64_t>(pm) * g.cl.s_pos + e;
                dst[0] = __float2bfloat16_rn(x1);
                dst[g.half] = __float2bfloat16_rn(x2);
            }
        }
    } else if (MODE == M_GU) {
        for (int idx = tid; idx < n * 64; idx += G_THREADS) {
            const int m = idx >> 6, u = idx & 63;
            const float rs = row_scale(g, m);
            const float gate = part_sum(g, m, c0 + u) * rs, up = part_sum(g, m, c0 + 64 + u) * rs;
            const float a = gate / (1.0f + expf(-gate)) * up;
            g.act[static_cast<int64_t>(m) * g.d_ff + 64 * t + u] = __float2bfloat16_rn(a);
        }
    } else {   // M_O, M_DOWN: residual update
        for (int idx = tid; idx < n * GT_N; idx += G_THREADS) {
            const int m = idx / GT_N, c = idx % GT_N;   // a warp: one item, 32 columns
            const int col = c0 + c;
            float* rp = g.resid + static_cast<int64_t>(m) * g.d + col;
            const float v = *rp + part_sum(g, m, col);
            *rp = v;
            if (g.h_out) {
                if (g.ipos[m] >= 0) g.h_out[static_cast<int64_t>(m) * g.ld_out + col] = __float2bfloat16_rn(v);
            } else {
                g.next_a[static_cast<int64_t>(m) * g.d + col] = __float2bfloat16_rn(v * __bfloat162float(g.next_gain[col]));
                const float sq = warp_sum(v * v);
                if ((threadIdx.x & 31) == 0) atomicAdd(g.ss_out + m, sq);
            }
        }
    }
    (void)ws;
}

template <int MODE>
__global__ void __launch_bounds__(G_THREADS, 1) w4_gemm_kernel(const __grid_constant__ GemmArgs g, void* ws) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* mma_bar = reinterpret_cast<uint64_t*>(smem + G_OFF_BAR);   // [2]
    uint64_t* acc_bar = mma_bar + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_bar + 1);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    __shared__ int s_last;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t = blockIdx.x, sp = blockIdx.y;
    const int n = item_count(g.n_max, g.n_dev);
    if (g.ss_zero && t == 0 && sp == 0)
        for (int i = tid; i < g.n_max; i += G_THREADS) g.ss_zero[i] = 0.f;
    if (n == 0) return;
    const int kc = g.K / g.ks, k0 = sp * kc, nkb = kc / GT_K;

    if (tid == 0) {
        tc::mbar_init(&mma_bar[0], 1);
        tc::mbar_init(&mma_bar[1], 1);
        tc::mbar_init(acc_bar, 1);
        *abort = 0;
        tc::fence_barrier_init();
    }
    if (warp == 0) tc::tmem_alloc(tmem_slot, GT_N);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // this thread's pieces of a block: one 16-byte code chunk (packed row tid / 8,
    // columns 16 (tid % 8) ...), and for tid < 32 one scale / zero chunk
    const int c_row = tid >> 3, c_chunk = tid & 7;
    int c_seg, c_col;
    tile_col<MODE>(g, t, c_chunk * 16, c_seg, c_col);
    const uint8_t* c_src = g.seg[c_seg].codes + static_cast<int64_t>(k0 / 2 + c_row) * g.seg[c_seg].n + c_col;
    const int64_t c_step = static_cast<int64_t>(GT_K / 2) * g.seg[c_seg].n;
    int z_seg = 0, z_col = 0;
    const bool z_thread = tid < 32;
    if (z_thread) tile_col<MODE>(g, t, (tid & 15) * 8, z_seg, z_col);
    const __half* z_src = (tid < 16 ? g.seg[z_seg].scale : g.seg[z_seg].zero) +
                          static_cast<int64_t>(k0 / GT_K) * g.seg[z_seg].n + z_col;
    const int64_t z_step = g.seg[z_seg].n;

    auto load_codes = [&](int kb) {
        if (kb >= nkb) return;
        const int st = kb % G_CS;
        cp_async16(smem + G_OFF_C + st * G_C_BYTES + c_row * GT_N + c_chunk * 16, c_src + kb * c_step);
        if (z_thread) cp_async16(smem + G_OFF_SZ + st * G_SZ_BYTES + tid * 16, z_src + kb * z_step);
    };
    auto load_a = [&](int kb) {
        if (kb >= nkb) return;
        uint8_t* dst = smem + G_OFF_A + (kb % G_AS) * G_A_BYTES;
        const bf16* src = g.a + k0 + kb * GT_K;
        for (int c = tid; c < n * 8; c += G_THREADS) {
            const int m = c >> 3, j = c & 7;
            cp_async16(dst + m * 128 + ((j ^ (m & 7)) << 4), src + static_cast<int64_t>(m) * g.lda + 8 * j);
        }
    };

    // prologue: codes of blocks 0 .. CS-2 and A of block 0 (one group), A of block 1
    for (int kb = 0; kb < G_CS - 1; ++kb) load_codes(kb);
    load_a(0);
    cp_commit();
    load_a(1);
    cp_commit();

    const int dq_n = tid & 127, dq_h = tid >> 7;   // dequantiser: column, half of the k block
    const uint32_t idesc = tc::idesc_bf16(128, GT_N);
    bool ok = true;
    for (int kb = 0; kb < nkb; ++kb) {
        if (tid == 0 && kb >= 2) {
            if (!tc::mbar_wait(&mma_bar[kb & 1], ((kb - 2) >> 1) & 1, abort, ws, 81)) *abort = 1;
        }
        __syncthreads();   // MMA kb-2 finished: its A stage and this B buffer are free
        if (*abort) {
            ok = false;
            break;
        }
        load_codes(kb + G_CS - 1);
        load_a(kb + 2);
        cp_commit();
        cp_wait<2>();      // block kb's codes and A have landed (this thread's copies)
        fence_async_smem();
        __syncthreads();
        {
            const uint8_t* cs = smem + G_OFF_C + (kb % G_CS) * G_C_BYTES;
            const __half* sz = reinterpret_cast<const __half*>(smem + G_OFF_SZ + (kb % G_CS) * G_SZ_BYTES);
            const float s = __half2float(sz[dq_n]);
            const float zs = -__half2float(sz[GT_N + dq_n]) * s;
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const uint32_t b = cs[(dq_h * 16 + i) * GT_N + dq_n];
                w[i] = pack_bf16x2(fmaf(static_cast<float>(b & 15u), s, zs), fmaf(static_cast<float>(b >> 4), s, zs));
            }
            uint8_t* row = smem + G_OFF_B + (kb & 1) * G_B_BYTES + dq_n * 128;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int jj = dq_h * 4 + q;
                *reinterpret_cast<uint4*>(row + ((jj ^ (dq_n & 7)) << 4)) =
                    make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
            }
        }
        fence_async_smem();
        __syncthreads();
        if (tid == 0) {
            tc::tc_fence_after();
            const uint64_t ad = tc::smem_desc_sw128(tc::smem_u32(smem + G_OFF_A + (kb % G_AS) * G_A_BYTES));
            const uint64_t bd = tc::smem_desc_sw128(tc::smem_u32(smem + G_OFF_B + (kb & 1) * G_B_BYTES));
#pragma unroll
            for (int kk = 0; kk < GT_K / 16; ++kk) tc::umma_bf16(tmem, ad + 2 * kk, bd + 2 * kk, idesc, kb | kk);
            tc::umma_commit(&mma_bar[kb & 1]);
        }
    }
    if (tid == 0) {
        tc::umma_commit(acc_bar);   // every MMA issued has finished (also after a stop)
        if (!tc::mbar_wait(acc_bar, 0, abort, ws, 82)) *abort = 1;
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    ok = ok && !*abort;
    tc::tc_fence_after();
    // partial tile -> workspace: warp w reads lanes 32 (w % 4).., columns 64 (w / 4)..
    if (ok) {
        const int m = (warp & 3) * 32 + lane;
        const int cb = (warp >> 2) * 64;
#pragma unroll 1
        for (int c = 0; c < 64; c += 32) {
            float v[32];
            tc::tmem_ld32(tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + cb + c, v);
            if (m < n) {
                float4* dst = reinterpret_cast<float4*>(g.part + (static_cast<int64_t>(sp) * g.n_max + m) * g.N +
                                                        t * GT_N + cb + c);
#pragma unroll
                for (int q = 0; q < 8; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            }
        }
    }
    tc::tc_fence_before();
    __threadfence();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, GT_N);
    if (!ok) return;
    if (tid == 0) {
        const int prev = atomicAdd(g.cnt + t, 1);
        s_last = prev == g.ks - 1;
        if (s_last) g.cnt[t] = 0;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    finish_tile<MODE>(g, t, n, ws);
}

// ------------------------------------------------------------------ attention
struct AttnArgs {
    int n_max;
    const int32_t* n_dev;
    int n_kv, qw, chunks;
    const bf16* qbuf;
    const int32_t* ipos;
    const int32_t* iseq;
    const bf16* kc;
    const bf16* vc;
    tee_cache_layout cl;
    int layer;
    float qscale;          // log2(e) / sqrt(head_dim)
    float* part;           // [n][n_kv][chunks][REP][HD + 2]
    int32_t* cnt;          // [n][n_kv]
    bf16* obuf;            // [n][qw]
};

constexpr int AT_THREADS = 128;

template <int HD, int REP>
__global__ void __launch_bounds__(AT_THREADS) river_attn_kernel(const __grid_constant__ AttnArgs a) {
    constexpr int RPT = 128 / HD;                 // K rows per thread in the score pass
    constexpr int CHUNK = AT_THREADS * RPT;       // positions per CTA
    constexpr int PC = HD / 8;                    // 16-byte pieces per row
    constexpr int RG = AT_THREADS / PC;           // row groups of the P.V pass
    __shared__ float s_q[REP][HD];
    __shared__ float s_p[REP][CHUNK];
    __shared__ float s_red[RG][REP][HD];
    __shared__ float s_mx[REP][AT_THREADS / 32], s_l[REP][AT_THREADS / 32];
    __shared__ float s_m[REP], s_sum[REP];
    __shared__ int s_last;

    const int c = blockIdx.x, g = blockIdx.y, m = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = item_count(a.n_max, a.n_dev);
    if (m >= n) return;
    const int pm = a.ipos[m];
    bf16* out = a.obuf + static_cast<int64_t>(m) * a.qw + static_cast<int64_t>(g) * REP * HD;
    if (pm < 0) {   // a skipped item attends to nothing
        if (c == 0)
            for (int i = tid; i < REP * HD; i += AT_THREADS) out[i] = __float2bfloat16_rn(0.f);
        return;
    }
    const int nch = pm / CHUNK + 1;
    if (c >= nch) return;
    const int t0 = c * CHUNK, cnt = min(CHUNK, pm + 1 - t0);
    const int64_t base = a.layer * a.cl.s_layer + a.iseq[m] * a.cl.s_seq + static_cast<int64_t>(g) * a.cl.s_head +
                         static_cast<int64_t>(t0) * a.cl.s_pos;
    for (int i = tid; i < REP * HD; i += AT_THREADS)
        s_q[i / HD][i % HD] = __bfloat162float(a.qbuf[static_cast<int64_t>(m) * a.qw + g * REP * HD + i]) * a.qscale;
    __syncthreads();

    // scores: thread -> RPT rows; every load of the rows issued before the sums
    float mx[REP];
#pragma unroll
    for (int r = 0; r < REP; ++r) mx[r] = -INFINITY;
    {
        uint4 kr[RPT][PC];
#pragma unroll
        for (int j = 0; j < RPT; ++j) {
            const int tt = tid + j * AT_THREADS;
            if (tt < cnt) {
                const uint4* src = reinterpret_cast<const uint4*>(a.kc + base + static_cast<int64_t>(tt) * a.cl.s_pos);
#pragma unroll
                for (int q = 0; q < PC; ++q) kr[j][q] = __ldcs(src + q);
            }
        }
#pragma unroll
        for (int j = 0; j < RPT; ++j) {
            const int tt = tid + j * AT_THREADS;
            if (tt >= cnt) continue;
            float acc[REP];
#pragma unroll
            for (int r = 0; r < REP; ++r) acc[r] = 0.f;
#pragma unroll
            for (int q = 0; q < PC; ++q) {
                float k8[8];
                unpack_bf16x2(kr[j][q].x, k8[0], k8[1]);
                unpack_bf16x2(kr[j][q].y, k8[2], k8[3]);
                unpack_bf16x2(kr[j][q].z, k8[4], k8[5]);
                unpack_bf16x2(kr[j][q].w, k8[6], k8[7]);
#pragma unroll
                for (int r = 0; r < REP; ++r)
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[r] = fmaf(s_q[r][8 * q + e], k8[e], acc[r]);
            }
#pragma unroll
            for (int r = 0; r < REP; ++r) {
                s_p[r][tt] = acc[r];
                mx[r] = fmaxf(mx[r], acc[r]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < REP; ++r) {
        float v = mx[r];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
        if (lane == 0) s_mx[r][warp] = v;
    }
    __syncthreads();
    if (tid < REP) {
        float v = -INFINITY;
        for (int w = 0; w < AT_THREADS / 32; ++w) v = fmaxf(v, s_mx[tid][w]);
        s_m[tid] = v;
    }
    __syncthreads();
    {
        float ls[REP];
#pragma unroll
        for (int r = 0; r < REP; ++r) ls[r] = 0.f;
#pragma unroll
        for (int j = 0; j < RPT; ++j) {
            const int tt = tid + j * AT_THREADS;
            if (tt >= cnt) continue;
#pragma unroll
            for (int r = 0; r < REP; ++r) {
                const float p = exp2f(s_p[r][tt] - s_m[r]);
                s_p[r][tt] = p;
                ls[r] += p;
            }
        }
#pragma unroll
        for (int r = 0; r < REP; ++r) {
            const float v = warp_sum(ls[r]);
            if (lane == 0) s_l[r][warp] = v;
        }
    }
    __syncthreads();
    if (tid < REP) {
        float v = 0.f;
        for (int w = 0; w < AT_THREADS / 32; ++w) v += s_l[tid][w];
        s_sum[tid] = v;
    }
    // P.V: thread (row group rg, piece pc): rows rg, rg + RG, ...; 8 columns
    {
        const int rg = tid / PC, pc = tid % PC;
        float o[REP][8];
#pragma unroll
        for (int r = 0; r < REP; ++r)
#pragma unroll
            for (int e = 0; e < 8; ++e) o[r][e] = 0.f;
        constexpr int ROWS = CHUNK / RG;
        constexpr int BATCH = 8;
#pragma unroll 1
        for (int b0 = 0; b0 < ROWS; b0 += BATCH) {
            uint4 vr[BATCH];
#pragma unroll
            for (int j = 0; j < BATCH; ++j) {
                const int tt = rg + (b0 + j) * RG;
                if (tt < cnt)
                    vr[j] = __ldcs(reinterpret_cast<const uint4*>(a.vc + base + static_cast<int64_t>(tt) * a.cl.s_pos) + pc);
            }
#pragma unroll
            for (int j = 0; j < BATCH; ++j) {
                const int tt = rg + (b0 + j) * RG;
                if (tt >= cnt) continue;
                float v8[8];
                unpack_bf16x2(vr[j].x, v8[0], v8[1]);
                unpack_bf16x2(vr[j].y, v8[2], v8[3]);
                unpack_bf16x2(vr[j].z, v8[4], v8[5]);
                unpack_bf16x2(vr[j].w, v8[6], v8[7]);
#pragma unroll
                for (int r = 0; r < REP; ++r) {
                    const float p = s_p[r][tt];
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[r][e] = fmaf(p, v8[e], o[r][e]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < REP; ++r)
#pragma unroll
            for (int e = 0; e < 8; ++e) s_red[rg][r][8 * pc + e] = o[r][e];
    }
    __syncthreads();
    if (nch == 1) {   // the whole range in this CTA: normalise and store
        for (int i = tid; i < REP * HD; i += AT_THREADS) {
            const int r = i / HD, e = i % HD;
            float v = 0.f;
            for (int w = 0; w < RG; ++w) v += s_red[w][r][e];
            out[i] = __float2bfloat16_rn(v / s_sum[r]);
        }
        return;
    }
    float* pp = a.part + ((static_cast<int64_t>(m) * a.n_kv + g) * a.chunks + c) * (REP * (HD + 2));
    for (int i = tid; i < REP * HD; i += AT_THREADS) {
        const int r = i / HD, e = i % HD;
        float v = 0.f;
        for (int w = 0; w < RG; ++w) v += s_red[w][r][e];
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
    // merge the chunks: O = sum_c o_c 2^(m_c - M) / sum_c l_c 2^(m_c - M)
    const float* p0 = a.part + (static_cast<int64_t>(m) * a.n_kv + g) * a.chunks * (REP * (HD + 2));
    for (int i = tid; i < REP * HD; i += AT_THREADS) {
        const int r = i / HD, e = i % HD;
        float M = -INFINITY;
        for (int cc = 0; cc < nch; ++cc) M = fmaxf(M, __ldcg(p0 + cc * (REP * (HD + 2)) + r * (HD + 2) + HD));
        float L = 0.f, O = 0.f;
        for (int cc = 0; cc < nch; ++cc) {
            const float* q = p0 + cc * (REP * (HD + 2)) + r * (HD + 2);
            const float w = exp2f(__ldcg(q + HD) - M);
            L = fmaf(__ldcg(q + HD + 1), w, L);
            O = fmaf(__ldcg(q + e), w, O);
        }
        out[i] = __float2bfloat16_rn(O / L);
    }
}

template <int HD>
tee_status launch_attn(const AttnArgs& a, int rep, dim3 grid, cudaStream_t s) {
    switch (rep) {
        case 1: river_attn_kernel<HD, 1><<<grid, AT_THREADS, 0, s>>>(a); break;
        case 2: river_attn_kernel<HD, 2><<<grid, AT_THREADS, 0, s>>>(a); break;
        case 4: river_attn_kernel<HD, 4><<<grid, AT_THREADS, 0, s>>>(a); break;
        case 8: river_attn_kernel<HD, 8><<<grid, AT_THREADS, 0, s>>>(a); break;
        default: return TEE_ERR_UNSUPPORTED;
    }
    return launch_status();
}

// ------------------------------------------------------------------ host
tee_status check_desc(const tee_river_desc* D) {
    if (!D) return TEE_ERR_INVALID_ARG;
    if (D->d <= 0 || D->n_q_heads <= 0 || D->n_kv_heads <= 0 || D->d_ff <= 0 || D->flags != 0)
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

template <int MODE>
tee_status launch_gemm(const GemmArgs& g, cudaStream_t s) {
    static bool attr = false;
    if (!attr) {
        tee_status st = cuda_status(cudaFuncSetAttribute(w4_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                         static_cast<int>(G_SMEM)));
        if (st != TEE_OK) return st;
        attr = true;
    }
    const int tiles = g.N / GT_N;
    w4_gemm_kernel<MODE><<<dim3(tiles, g.ks), G_THREADS, G_SMEM, s>>>(g, nullptr);
    return launch_status();
}

}  // namespace

}  // namespace tee

using namespace tee;

extern "C" size_t tee_exit_river_prep_size(const tee_river_desc* D, int32_t max_pos) {
    if (check_desc(D) != TEE_OK || max_pos <= 0) return 0;
    return PREP_HEADER_BYTES + rope_table_bytes(max_pos, D->head_dim);
}

extern "C" tee_status tee_exit_river_prepare(const tee_river_desc* D, int32_t max_pos, void* prep, size_t prep_bytes,
                                             void* stream) {
    tee_status st = check_desc(D);
    if (st != TEE_OK) return st;
    if (max_pos <= 0) return TEE_ERR_INVALID_ARG;
    if (!prep || !aligned16(prep) || prep_bytes < tee_exit_river_prep_size(D, max_pos)) return TEE_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    PrepHeader h{};
    h.magic = RIVER_MAGIC;
    h.d = D->d;
    h.n_kv_heads = D->n_kv_heads;
    h.head_dim = D->head_dim;
    h.max_pos = max_pos;
    st = cuda_status(cudaMemcpyAsync(prep, &h, sizeof(h), cudaMemcpyHostToDevice, s));
    if (st != TEE_OK) return st;
    float2* table = reinterpret_cast<float2*>(static_cast<char*>(prep) + PREP_HEADER_BYTES);
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
        if (!seg_ok(L.wq) || !seg_ok(L.wk) || !seg_ok(L.wv) || !seg_ok(L.wo) || !seg_ok(L.wg) || !seg_ok(L.wu) ||
            !seg_ok(L.wd))
            return TEE_ERR_INVALID_ARG;
        if (L.cache_layer < 0 || L.cache_layer >= cl.n_layers) return TEE_ERR_INVALID_ARG;
    }
    if (!prep || !aligned16(prep) || prep_bytes < PREP_HEADER_BYTES + sizeof(float2) * (hd / 2))
        return TEE_ERR_WORKSPACE;
    const RiverWs w = river_ws(*D, n_max, cl.max_pos);
    if (!ws || ws_bytes < w.end) return TEE_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const PrepHeader* hdr = static_cast<const PrepHeader*>(prep);
    const float2* rope = reinterpret_cast<const float2*>(static_cast<const char*>(prep) + PREP_HEADER_BYTES);

    float* resid = ws_at<float>(ws, w.resid);
    bf16* abuf = ws_at<bf16>(ws, w.abuf);
    bf16* qbuf = ws_at<bf16>(ws, w.qbuf);
    bf16* obuf = ws_at<bf16>(ws, w.obuf);
    bf16* act = ws_at<bf16>(ws, w.act);
    float* ss_a = ws_at<float>(ws, w.ss_a);
    float* ss_f = ws_at<float>(ws, w.ss_f);
    int32_t* ipos = ws_at<int32_t>(ws, w.ipos);
    int32_t* iseq = ws_at<int32_t>(ws, w.iseq);
    int32_t* gcnt = ws_at<int32_t>(ws, w.gcnt);
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
    ga.cnt = gcnt;
    ga.n_cnt = static_cast<int>((w.acnt - w.gcnt) / 4 + static_cast<size_t>(n_max) * D->n_kv_heads);
    river_gather_kernel<<<n_max, 256, 0, s>>>(ga, ws);
    if ((st = launch_status()) != TEE_OK) return st;

    GemmArgs g{};
    g.n_max = n_max;
    g.n_dev = n_dev;
    g.part = ws_at<float>(ws, w.part);
    g.cnt = gcnt;
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
    at.chunks = (cl.max_pos + at_chunk(hd) - 1) / at_chunk(hd);
    at.qbuf = qbuf;
    at.ipos = ipos;
    at.iseq = iseq;
    at.kc = static_cast<const bf16*>(k_cache);
    at.vc = static_cast<const bf16*>(v_cache);
    at.cl = cl;
    at.qscale = 1.4426950408889634f / sqrtf(static_cast<float>(hd));
    at.part = ws_at<float>(ws, w.apart);
    at.cnt = acnt;
    at.obuf = obuf;
    const int rep = D->n_q_heads / D->n_kv_heads;

    for (int l = 0; l < n_layers; ++l) {
        const tee_river_layer& L = layers[l];
        const bool last = l == n_layers - 1;
        // q | k | v
        g.seg[0] = seg_of(L.wq, qw);
        g.seg[1] = seg_of(L.wk, kvw);
        g.seg[2] = seg_of(L.wv, kvw);
        g.n_seg = 3;
        g.K = d;
        g.N = qw + 2 * kvw;
        g.ks = choose_ks(g.N / GT_N, d);
        g.a = abuf;
        g.lda = d;
        g.ss_in = ss_a;
        g.inv_width = 1.0f / d;
        g.ss_zero = nullptr;
        g.layer = L.cache_layer;
        if ((st = launch_gemm<M_QKV>(g, s)) != TEE_OK) return st;
        // attention
        at.layer = L.cache_layer;
        const dim3 agrid(at.chunks, D->n_kv_heads, n_max);
        st = hd == 64 ? launch_attn<64>(at, rep, agrid, s) : launch_attn<128>(at, rep, agrid, s);
        if (st != TEE_OK) return st;
        // h1 = h + o Wo
        g.seg[0] = seg_of(L.wo, d);
        g.n_seg = 1;
        g.K = qw;
        g.N = d;
        g.ks = choose_ks(d / GT_N, qw);
        g.a = obuf;
        g.lda = qw;
        g.ss_in = nullptr;
        g.next_gain = static_cast<const bf16*>(L.ffn_norm);
        g.next_a = abuf;
        g.ss_out = ss_f;
        g.h_out = nullptr;
        if ((st = launch_gemm<M_O>(g, s)) != TEE_OK) return st;
        // a = SiLU(x2 Wg) * (x2 Wu)
        g.seg[0] = seg_of(L.wg, f);
        g.seg[1] = seg_of(L.wu, f);
        g.n_seg = 2;
        g.K = d;
        g.N = 2 * f;
        g.ks = choose_ks(g.N / GT_N, d);
        g.a = abuf;
        g.lda = d;
        g.ss_in = ss_f;
        g.ss_zero = ss_a;
        if ((st = launch_gemm<M_GU>(g, s)) != TEE_OK) return st;
        // h2 = h1 + a Wd
        g.seg[0] = seg_of(L.wd, d);
        g.n_seg = 1;
        g.K = f;
        g.N = d;
        g.ks = choose_ks(d / GT_N, f);
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
        if ((st = launch_gemm<M_DOWN>(g, s)) != TEE_OK) return st;
    }
    return TEE_OK;
}
