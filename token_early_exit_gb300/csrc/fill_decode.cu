// Decode path of the KV fill: up to 128 items (decode tokens that exit), int4
// group-64 weights (River-LLM's W4A16 exit layers), identity map (the
// "State Propagation" / identity-fill input).
//
// Work split. The K and V projections of one filled layer are cut into groups
// of 256 output columns, and the reduction dimension d into KS equal ranges.
// One cluster of KS CTAs per (group, layer): CTA r computes, on tcgen05,
//   P_r[item][c] = sum_{k in range r} h[row(item)][k] * W'[k][c],
//   W'[k][c] = (q - zero) * scale * g_j[k]     (M = 128 item rows, N = 256, K = d / KS)
// and the partial sums of h^2 over its range; the CTAs then add their partials
// through the workspace (L2). A group is four units of 64 columns, each
// unit the two 32-wide halves [i, i+32) and [i+hd/2, i+hd/2+32) of one head,
// so that RoPE pairs stay inside a unit; unit u is finished by the CTA of rank
// u % KS: sum of the KS partials, 1/rms over the whole d, RoPE, bf16 store
// into the backbone's cache slot.
//
// Warp roles in a CTA (mbarriers between roles):
//   warps 0-7   stream the CTA's int4 codes and fp16 scales/zeros (cp.async, 256-k
//               chunks, two in flight) and dequantise each 64-k block into a ring
//               of bf16 B operands (256 rows of 128 bytes, 128-byte swizzle):
//               W'[k][c] = (q - z) s g_j[k], in packed bf16x2 arithmetic;
//   warp 8      issues tcgen05.mma (N = 256) into a 256-column TMEM accumulator;
//   warps 9-12  gather the items' h rows of each 64-k block into a ring of A
//               operands (cp.async, 128-byte swizzle), after asking L2 for the
//               rows' slices at the start. Once a thread's pieces of a block have
//               landed it adds their squares into per-item sums of h^2 and
//               releases the block; they also fetch positions and cache slots.
// After the last MMA warps 0-7 store the accumulator rows (thread = item row,
// TMEM lane quarter = warp % 4) and the partial sums of h^2 into this CTA's slot
// of the workspace with coalesced 16-byte stores; one cluster barrier (release /
// acquire at cluster scope); then warps 0-7 of each CTA read the KS partials of
// their units from L2, add them and finish.
#include "fill.cuh"
#include "tc.cuh"

namespace tee {

namespace {

using bf16 = __nv_bfloat16;

constexpr int D_GCOLS = 256;         // output columns per group (MMA N)
constexpr int D_UNITS = 4;           // 64-column units per group
constexpr int D_KB = 64;             // K per MMA block (one int4 group)
constexpr int D_CH = 256;            // K per staged chunk of codes
constexpr int D_BPC = D_CH / D_KB;   // blocks per chunk
constexpr int D_RA = 5;              // A operand slots (h rows)
constexpr int D_LAG = 2;             // blocks of h copies in flight
constexpr int D_RC = 2;              // code chunks in flight
constexpr int D_MAX_ITEMS = 128;
constexpr int D_DEQ_WARPS = 8, D_MMA_WARP = 8, D_CP_WARP0 = 9, D_CP_WARPS = 4;
constexpr int D_DEQ_THREADS = D_DEQ_WARPS * 32;
constexpr int D_CP_THREADS = D_CP_WARPS * 32;
constexpr int D_THREADS = (D_CP_WARP0 + D_CP_WARPS) * 32;
constexpr int D_MAX_KC = 2048;       // largest k range of one CTA (its g_j slice sits in shared memory)
// A slot is refilled D_RA - D_LAG - 1 iterations after its release: slack for the
// MMA round trip (an mbarrier hand-off costs ~0.1 us).
static_assert(D_LAG + 2 < D_RA, "the A ring needs slack beyond the blocks in flight");

constexpr uint32_t B_SLOT = D_GCOLS * 128;              // 32 KB: 256 columns x 64 k
constexpr uint32_t CH_CODES = (D_CH / 2) * D_GCOLS;     // 32 KB: 128 packed rows x 256 columns
constexpr uint32_t CH_SZ = (D_CH / D_KB) * D_GCOLS * 4; // 4 KB: scale[256], zero[256] (fp16) per group
constexpr uint32_t CH_BYTES = CH_CODES + CH_SZ;

// Shared-memory layout. Up to 128 items the A slots hold 128 item rows and the B
// ring two dequantised blocks. Up to 64 items ("narrow") the A slots hold 64 rows:
// the M = 128 MMA then also reads the next 64 rows (the following slot, or after
// the last slot an 8 KB guard), which only feed accumulator rows >= 64 that are
// never stored; the space saved gives the B ring a third slot, so that the
// dequantising warps do not wait for the MMA of two blocks back.
template <bool NARROW>
struct DLayout {
    static constexpr int ITEMS = NARROW ? 64 : 128;
    static constexpr int RB = NARROW ? 3 : 2;             // B operand slots (dequantised weights)
    static constexpr uint32_t A_SLOT = ITEMS * 128;       // item rows x 64 k
    static constexpr uint32_t A_GUARD = NARROW ? 64 * 128 : 0;
    static constexpr uint32_t OFF_A = 0;
    static constexpr uint32_t OFF_B = OFF_A + D_RA * A_SLOT + A_GUARD;
    static constexpr uint32_t OFF_C = OFF_B + RB * B_SLOT;
    static constexpr uint32_t OFF_G = OFF_C + D_RC * CH_BYTES;    // g_j over this CTA's k range (bf16)
    static constexpr uint32_t OFF_SMALL = OFF_G + D_MAX_KC * 2;
    static constexpr uint32_t SMALL_BYTES = (2 * D_RA + 2 * RB + 2) * 8 + D_MAX_ITEMS * (8 + 4 + 4) + 16;
    static constexpr size_t SMEM = 1024 + OFF_SMALL + SMALL_BYTES;
    static constexpr int IPC = ITEMS * 8 / D_CP_THREADS;  // 16-byte h pieces per copy thread and block
    static_assert(SMEM <= 232448, "decode fill shared memory");
    static_assert(OFF_B % 1024 == 0 && OFF_C % 16 == 0 && OFF_G % 16 == 0 && OFF_SMALL % 8 == 0, "alignment");
};

struct DecodeLayer {
    const uint8_t* codes[2];   // wk, wv
    const __half* scale[2];
    const __half* zero[2];
    const bf16* gamma;
    const bf16* bias[2];   // k_bias, v_bias (nullable)
    const bf16* k_norm;    // per-head K norm weight (nullable)
    int cache_layer;
    int writes;            // 0, TEE_FILL_WRITE_K or TEE_FILL_WRITE_V
};
constexpr int MAX_DECODE_LAYERS = 64;
struct DecodeArgs {
    DecodeLayer l[MAX_DECODE_LAYERS];
    int n_max, d, kvw, hd, half, groups_kv, ks;
    const int32_t* n_dev;
    float inv_d, eps;
    const bf16* h;
    int64_t ld_h;
    int h_rows;
    const int32_t* rows;
    const int32_t* pos;
    int pos0;
    const int32_t* seq;
    const PrepHeader* hdr;
    const float2* rope;
    bf16* kc;
    bf16* vc;
    tee_cache_layout cl;
    float4* part;   // workspace: [cluster][rank][unit][16][n_max] float4 partial accumulators
    float* part_ss; // workspace: [cluster][rank][n_max] partial sums of h^2
};

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(tc::smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void deq_bar_sync() {   // the eight dequantising warps only
    asm volatile("bar.sync 1, %0;" ::"n"(D_DEQ_THREADS) : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
// Lane 0 waits for the phase, the warp follows: every lane sees the same outcome,
// so a timed-out wait cannot split a warp at a later __syncwarp or named barrier.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort, void* ws, int where) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = tc::mbar_wait(bar, parity, abort, ws, where);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    __syncwarp();
    return ok;
}
__device__ __forceinline__ float sumsq8(uint4 x, float acc) {
    float f[8];
    unpack_bf16x2(x.x, f[0], f[1]);
    unpack_bf16x2(x.y, f[2], f[3]);
    unpack_bf16x2(x.z, f[4], f[5]);
    unpack_bf16x2(x.w, f[6], f[7]);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc = fmaf(f[e], f[e], acc);
    return acc;
}
// Two consecutive k of one column from byte b of a packed word (low nibble = the
// lower k): x = (b & 0xF) | (b >> 4) << 16 | 0x43004300 is the bf16 pair 128 + q;
// subtracting 136 leaves q - 8 exactly, and one bf16x2 fma gives
// (q - 8) s + (8 - z) s = (q - z) s, rounded once, then the RMSNorm gains of the
// two k (rounded again). wl / wh: the packed word and the word shifted right by 4;
// sel picks byte b of each into bytes 0 and 2.
__device__ __forceinline__ uint32_t deq_pair(uint32_t wl, uint32_t wh, uint32_t sel, __nv_bfloat162 s2,
                                             __nv_bfloat162 zs2, __nv_bfloat162 g2) {
    const uint32_t x = (__byte_perm(wl, wh, sel) & 0x000F000Fu) | 0x43004300u;
    __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&x);
    v = __hmul2(__hfma2(__hsub2(v, __floats2bfloat162_rn(136.0f, 136.0f)), s2, zs2), g2);
    return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// L2-only loads of what peer CTAs wrote before the cluster barrier (that barrier's
// asm carries the memory clobber, so these cannot move above it).
__device__ __forceinline__ float4 ld_l2_f4(const float4* p) {
    float4 v;
    asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ float ld_l2_f32(const float* p) {
    float v;
    asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ void load8_bf16(const bf16* p, float (&v)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    unpack_bf16x2(u.x, v[0], v[1]);
    unpack_bf16x2(u.y, v[2], v[3]);
    unpack_bf16x2(u.z, v[4], v[5]);
    unpack_bf16x2(u.w, v[6], v[7]);
}

// One thread's 8 low and 8 high output columns (columns col, col + half of the
// projection): the partial accumulators of the ks split CTAs summed, times the
// row's 1/rms, plus the bias.
__device__ __forceinline__ void sum_partials(const float4 (&pv)[4][4], int ks, float rs, const bf16* bias, int col,
                                             int half, float (&lo)[8], float (&hi)[8]) {
#pragma unroll
    for (int e = 0; e < 8; ++e) lo[e] = hi[e] = 0.f;
#pragma unroll
    for (int src = 0; src < 4; ++src) {
        if (src >= ks) continue;
        const float4 l0 = pv[src][0], l1 = pv[src][1], h0 = pv[src][2], h1 = pv[src][3];
        lo[0] += l0.x; lo[1] += l0.y; lo[2] += l0.z; lo[3] += l0.w;
        lo[4] += l1.x; lo[5] += l1.y; lo[6] += l1.z; lo[7] += l1.w;
        hi[0] += h0.x; hi[1] += h0.y; hi[2] += h0.z; hi[3] += h0.w;
        hi[4] += h1.x; hi[5] += h1.y; hi[6] += h1.z; hi[7] += h1.w;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        lo[e] *= rs;
        hi[e] *= rs;
    }
    if (bias) {
        float b[8];
        load8_bf16(bias + col, b);
#pragma unroll
        for (int e = 0; e < 8; ++e) lo[e] += b[e];
        load8_bf16(bias + col + half, b);
#pragma unroll
        for (int e = 0; e < 8; ++e) hi[e] += b[e];
    }
}

// First column of unit u's low and high halves within the K (or V) projection.
__device__ __forceinline__ int unit_col_lo(int gk, int u, int hd) {
    const int uph = hd / 64;   // units per head
    return (D_GCOLS * gk / hd + u / uph) * hd + 32 * (u % uph);
}

template <bool NARROW>
__global__ void __launch_bounds__(D_THREADS, 1)
fill_decode_kernel(const __grid_constant__ DecodeArgs a, void* ws) {
    using Lay = DLayout<NARROW>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* a_full = reinterpret_cast<uint64_t*>(smem + Lay::OFF_SMALL);
    uint64_t* a_empty = a_full + D_RA;
    uint64_t* b_full = a_empty + D_RA;
    uint64_t* b_empty = b_full + Lay::RB;
    uint64_t* acc_full = b_empty + Lay::RB;
    uint64_t* ss_ready = acc_full + 1;
    int64_t* s_ioff = reinterpret_cast<int64_t*>(ss_ready + 1);   // item part of the cache offset, or -1
    int* s_pos = reinterpret_cast<int*>(s_ioff + D_MAX_ITEMS);
    float* s_ss = reinterpret_cast<float*>(s_pos + D_MAX_ITEMS);  // partial sum(h^2) over this CTA's k
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s_ss + D_MAX_ITEMS);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int ks = a.ks;
    const int rank = static_cast<int>(cluster_rank());
    const int gq = blockIdx.x / ks, li = blockIdx.y;
    const DecodeLayer& L = a.l[li];
    const bool is_k = gq < a.groups_kv;
    const int kv = is_k ? 0 : 1;
    const int gk = is_k ? gq : gq - a.groups_kv;
    // A K-only or V-only layer: the other kind's clusters leave before any shared state.
    if (L.writes == (is_k ? TEE_FILL_WRITE_V : TEE_FILL_WRITE_K)) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kc = a.d / ks, k0 = rank * kc;     // this CTA's k range
    const int nkb = kc / D_KB, nch = kc / D_CH;
    // The item count (and everything else a previous kernel may produce) is read only
    // after wait_prior_grid(): with an early launch the weights stream in before that.
    int n = 0;
    // one CTA (the first that runs for layer 0) records bad rows / positions
    const bool reporter = li == 0 && blockIdx.x == (a.l[0].writes == TEE_FILL_WRITE_V ? a.groups_kv * ks : 0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < D_RA; ++s) {
            tc::mbar_init(&a_full[s], D_CP_WARPS);
            tc::mbar_init(&a_empty[s], 1);                // MMA commit
        }
        for (int s = 0; s < Lay::RB; ++s) {
            tc::mbar_init(&b_full[s], D_DEQ_WARPS);
            tc::mbar_init(&b_empty[s], 1);
        }
        tc::mbar_init(acc_full, 1);
        tc::mbar_init(ss_ready, D_CP_WARPS);
        *abort = 0;
        tc::fence_barrier_init();
    }
    // Chunk c of the CTA's codes / scales / zeros into ring slot c % D_RC. Staged
    // column order: unit u's low half, then its high half (64 u .. 64 u + 63).
    // Per-thread pieces of a chunk (dequant warps): code piece p = t % 16 of packed
    // rows t / 16 + 16 i, and scale/zero piece t (group, which, unit, half, quarter).
    const int p_code = threadIdx.x & 15, r_code = threadIdx.x >> 4;
    const int col_code = unit_col_lo(gk, p_code >> 2, a.hd) + ((p_code & 3) >= 2 ? a.half : 0) + (p_code & 1) * 16;
    const int g_sz = (threadIdx.x >> 6) & 3, which_sz = (threadIdx.x >> 5) & 1, p_sz = threadIdx.x & 31;
    const int col_sz = unit_col_lo(gk, p_sz >> 3, a.hd) + (((p_sz >> 2) & 1) ? a.half : 0) + (p_sz & 3) * 8;
    const uint32_t off_sz = CH_CODES + g_sz * (D_GCOLS * 4) + which_sz * (D_GCOLS * 2) +
                            ((p_sz >> 3) * 64 + ((p_sz >> 2) & 1) * 32 + (p_sz & 3) * 8) * 2;
    // Chunk c of the CTA's codes / scales / zeros into ring slot c % D_RC. Staged
    // column order: unit u's low half, then its high half (64 u .. 64 u + 63).
    auto load_chunk = [&](int c) {
        uint8_t* base = smem + Lay::OFF_C + (c % D_RC) * CH_BYTES;
        const int kg = k0 + c * D_CH;             // first k of the chunk
        const uint8_t* src = L.codes[kv] + static_cast<int64_t>(kg / 2 + r_code) * a.kvw + col_code;
#pragma unroll
        for (int i = 0; i < (D_CH / 2) / 16; ++i)
            cp_async16(base + (r_code + 16 * i) * D_GCOLS + p_code * 16, src + static_cast<int64_t>(16 * i) * a.kvw);
        static_assert(D_BPC * 64 == D_DEQ_THREADS, "one scale/zero piece per thread");
        cp_async16(base + off_sz,
                   (which_sz ? L.zero[kv] : L.scale[kv]) + static_cast<int64_t>(kg / D_KB + g_sz) * a.kvw + col_sz);
    };
    if (warp < D_DEQ_WARPS) {
        // g_j over this CTA's k range rides in chunk 0's group.
        for (int v = threadIdx.x; v < kc / 8; v += D_DEQ_THREADS) cp_async16(smem + Lay::OFF_G + v * 16, L.gamma + k0 + v * 8);
        for (int c = 0; c < D_RC; ++c) {
            if (c < nch) load_chunk(c);
            cp_async_commit();
        }
    }
    if (warp == D_MMA_WARP) tc::tmem_alloc(tmem_slot, D_GCOLS);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < D_DEQ_WARPS) {
        // ---- dequantise. Thread t: staged columns 4 cg .. 4 cg + 3 (cg = t % 64), k
        // 16 kq .. 16 kq + 15 of each block (kq = t / 64). Staged column 4 cg + j goes
        // to B row (= accumulator column) cg + 64 j: consecutive lanes hit different
        // swizzle rows, so the 16-byte stores are conflict-free.
        const int t = threadIdx.x;
        const int cg = t & 63, kq = t >> 6;
        bool ok = true;
        for (int c = 0; c < nch; ++c) {
            cp_async_wait<D_RC - 1>();                            // chunk c has landed (own copies)
            deq_bar_sync();                                       // ... and everyone's
            const uint8_t* base = smem + Lay::OFF_C + (c % D_RC) * CH_BYTES;
            for (int b = 0; b < D_BPC && ok; ++b) {
                const int kb = c * D_BPC + b, s = kb % Lay::RB;
                if (kb >= Lay::RB && !warp_wait(&b_empty[s], ((kb / Lay::RB) - 1) & 1, abort, ws, 51)) {
                    ok = false;
                    break;
                }
                uint32_t w[8], wh[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    w[i] = *reinterpret_cast<const uint32_t*>(base + (b * 32 + kq * 8 + i) * D_GCOLS + 4 * cg);
                    wh[i] = w[i] >> 4;
                }
                const uint8_t* szp = base + CH_CODES + b * (D_GCOLS * 4);
                const uint2 s4 = *reinterpret_cast<const uint2*>(szp + cg * 8);
                const uint2 z4 = *reinterpret_cast<const uint2*>(szp + D_GCOLS * 2 + cg * 8);
                float sc[4], zr[4];
                unpack_f16x2(s4.x, sc[0], sc[1]);
                unpack_f16x2(s4.y, sc[2], sc[3]);
                unpack_f16x2(z4.x, zr[0], zr[1]);
                unpack_f16x2(z4.y, zr[2], zr[3]);
                // g_j of the thread's 16 k, as 8 bf16 pairs (k 16 kq + 2i, +1)
                const uint4 ga = *reinterpret_cast<const uint4*>(smem + Lay::OFF_G + (kb * D_KB + kq * 16) * 2);
                const uint4 gb = *reinterpret_cast<const uint4*>(smem + Lay::OFF_G + (kb * D_KB + kq * 16 + 8) * 2);
                const uint32_t gw[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
                uint8_t* bslot = smem + Lay::OFF_B + s * B_SLOT;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const __nv_bfloat162 s2 = __floats2bfloat162_rn(sc[j], sc[j]);
                    const float zs = (8.0f - zr[j]) * sc[j];
                    const __nv_bfloat162 zs2 = __floats2bfloat162_rn(zs, zs);
                    const uint32_t sel = (j | (j << 4) | ((j + 4) << 8) | ((j + 4) << 12));
                    uint32_t o[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)   // k 16 kq + 2i, +1
                        o[i] = deq_pair(w[i], wh[i], sel, s2, zs2, *reinterpret_cast<const __nv_bfloat162*>(&gw[i]));
                    const int row = cg + 64 * j;
                    uint8_t* rp = bslot + row * 128;
                    *reinterpret_cast<uint4*>(rp + (((2 * kq) ^ (row & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
                    *reinterpret_cast<uint4*>(rp + (((2 * kq + 1) ^ (row & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&b_full[s]);
            }
            deq_bar_sync();                                       // everyone is done with chunk c
            if (c + D_RC < nch) load_chunk(c + D_RC);
            cp_async_commit();
        }
    } else if (warp == D_MMA_WARP) {
        // ---- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_bf16(128, D_GCOLS);
            for (int kb = 0; kb < nkb; ++kb) {
                const int sa = kb % D_RA, sb = kb % Lay::RB;
                if (!tc::mbar_wait(&a_full[sa], (kb / D_RA) & 1, abort, ws, 53)) break;
                if (!tc::mbar_wait(&b_full[sb], (kb / Lay::RB) & 1, abort, ws, 54)) break;
                tc::tc_fence_after();
                const uint64_t ad = tc::smem_desc_sw128(tc::smem_u32(smem + Lay::OFF_A + sa * Lay::A_SLOT));
                const uint64_t bd = tc::smem_desc_sw128(tc::smem_u32(smem + Lay::OFF_B + sb * B_SLOT));
#pragma unroll
                for (int kk = 0; kk < D_KB / 16; ++kk) tc::umma_bf16(tmem, ad + 2 * kk, bd + 2 * kk, idesc, kb | kk);
                tc::umma_commit(&a_empty[sa]);
                tc::umma_commit(&b_empty[sb]);
            }
            tc::umma_commit(acc_full);   // also when stopped early: every issued MMA finishes first
        }
    } else {
        // ---- h rows. Thread ct copies 16-byte piece j = ct % 8 (k 8 j .. 8 j + 7 of
        // each block) of items ct / 8 + 16 m, m = 0..7, of every block of this CTA's
        // k range; it alone touches those pieces, so once they have landed it adds
        // their squares and scales them by g_j in place.
        const int ct = threadIdx.x - D_CP_WARP0 * 32;
        const int j = ct & 7, ib = ct >> 3;
        wait_prior_grid();
        n = min(item_count(a.n_max, a.n_dev), Lay::ITEMS);
        // Item ct's h row slice, pulled into L2 whole (every CTA of the column groups
        // reads it).
        int r_ct = -1;
        if (ct < n) {
            const int r = a.rows ? a.rows[ct] : ct;
            if (r >= 0 && r < a.h_rows) {
                r_ct = r;
                prefetch_l2(a.h + static_cast<int64_t>(r) * a.ld_h + k0, static_cast<uint32_t>(kc * 2));
            } else if (reporter) {
                record_fault(ws, TEE_DEVERR_ROW, r);
            }
        }
        const bf16* src[Lay::IPC];
#pragma unroll
        for (int m = 0; m < Lay::IPC; ++m) {
            const int i = ib + 16 * m;
            const int r = i < n ? (a.rows ? a.rows[i] : i) : -1;
            src[m] = (r >= 0 && r < a.h_rows) ? a.h + static_cast<int64_t>(r) * a.ld_h + k0 + j * 8 : nullptr;
        }
        auto issue = [&](int kb) {
            uint8_t* slot = smem + Lay::OFF_A + (kb % D_RA) * Lay::A_SLOT;
#pragma unroll
            for (int m = 0; m < Lay::IPC; ++m) {
                const int i = ib + 16 * m;
                if (src[m]) cp_async16(slot + i * 128 + ((j ^ (i & 7)) << 4), src[m] + kb * D_KB);
            }
        };
        float ss[Lay::IPC];
#pragma unroll
        for (int m = 0; m < Lay::IPC; ++m) ss[m] = 0.f;
        // Block kb's pieces of this thread have landed: add their squares, order them
        // for the tensor core, and release the block once the whole warp is done.
        auto release = [&](int kb) {
            const uint8_t* slot = smem + Lay::OFF_A + (kb % D_RA) * Lay::A_SLOT;
#pragma unroll
            for (int m = 0; m < Lay::IPC; ++m) {
                if (!src[m]) continue;
                const int i = ib + 16 * m;
                ss[m] = sumsq8(*reinterpret_cast<const uint4*>(slot + i * 128 + ((j ^ (i & 7)) << 4)), ss[m]);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&a_full[kb % D_RA]);
        };
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
            const int s = kb % D_RA;
            if (kb >= D_RA && !warp_wait(&a_empty[s], ((kb / D_RA) - 1) & 1, abort, ws, 52)) {
                ok = false;
                break;
            }
            issue(kb);
            cp_async_commit();
            if (kb >= D_LAG) {
                cp_async_wait<D_LAG>();
                release(kb - D_LAG);
            }
        }
        cp_async_wait<0>();
        if (ok)
            for (int b = max(0, nkb - D_LAG); b < nkb; ++b) release(b);
        // Per-item totals: the eight threads of an item are consecutive lanes.
#pragma unroll
        for (int m = 0; m < Lay::IPC; ++m) {
            float t = ss[m];
            t += __shfl_xor_sync(0xffffffffu, t, 1);
            t += __shfl_xor_sync(0xffffffffu, t, 2);
            t += __shfl_xor_sync(0xffffffffu, t, 4);
            if (j == 0) s_ss[ib + 16 * m] = t;
        }
        // Item ct's position and cache slot (dependent loads: kept off the copies' path).
        {
            int64_t ioff = -1;
            int p = 0;
            if (r_ct >= 0) {
                p = a.pos ? a.pos[r_ct] : a.pos0 + r_ct;
                const int sq = a.seq ? a.seq[r_ct] : 0;
                if (!pos_ok(p, a.cl.max_pos, a.hdr)) {
                    if (reporter) record_fault(ws, TEE_DEVERR_POS, p);
                    p = 0;
                } else if (sq < 0 || sq >= a.cl.n_seq) {
                    if (reporter) record_fault(ws, TEE_DEVERR_SEQ, sq);
                } else {
                    ioff = L.cache_layer * a.cl.s_layer + sq * a.cl.s_seq + static_cast<int64_t>(p) * a.cl.s_pos;
                    if (is_k) prefetch_l2(a.rope + static_cast<int64_t>(p) * a.half, static_cast<uint32_t>(a.half * 8));
                }
            }
            s_ioff[ct] = ioff;
            s_pos[ct] = p;
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(ss_ready);   // release: s_ss, s_ioff, s_pos are ready
    }

    wait_prior_grid();
    n = min(item_count(a.n_max, a.n_dev), Lay::ITEMS);
    // ---- the reduction across the cluster, through this call's workspace slots.
    // Accumulator column cg + 64 j holds staged column 4 cg + j, i.e. unit cg / 16,
    // unit column 4 (cg % 16) + j: float4 m = cg % 16 of a unit row holds its
    // unit columns 4m .. 4m + 3.
    const int cluster = blockIdx.y * (gridDim.x / ks) + gq;
    float4* part = a.part + static_cast<int64_t>(cluster) * ks * D_UNITS * 16 * a.n_max;
    float* part_ss = a.part_ss + static_cast<int64_t>(cluster) * ks * a.n_max;
    bool acc_ok = true;
    if (warp < D_DEQ_WARPS) {
        acc_ok = warp_wait(acc_full, 0, abort, ws, 56);
        acc_ok = warp_wait(ss_ready, 0, abort, ws, 57) && acc_ok;   // s_ss, s_ioff, s_pos
        tc::tc_fence_after();
        // Warp w reads TMEM lane quarter w % 4 (item rows 32 (w % 4) + lane), units
        // 2 (w / 4) and 2 (w / 4) + 1; consecutive lanes store consecutive rows.
        const int r = (warp & 3) * 32 + lane;
        const uint32_t tb = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
#pragma unroll 1
        for (int u = 2 * (warp >> 2); u < 2 * (warp >> 2) + 2; ++u) {
            float v[4][16];
            tc::tmem_ld16x4(tb + 16 * u, 64, v);   // warp-wide
            if (acc_ok && r < n) {
                float4* dst = part + static_cast<int64_t>((rank * D_UNITS + u) * 16) * a.n_max + r;
#pragma unroll
                for (int m = 0; m < 16; ++m) dst[static_cast<int64_t>(m) * a.n_max] = make_float4(v[0][m], v[1][m], v[2][m], v[3][m]);
            }
        }
        if (warp < 4 && acc_ok && r < n) part_ss[rank * a.n_max + r] = s_ss[r];
    }
    tc::tc_fence_before();
    cluster_sync();   // every CTA's partials are visible to the cluster
    tc::tc_fence_after();

    // ---- finish the units of this rank: warps 0-7, thread = (item, 8 column pairs).
    if (warp < D_DEQ_WARPS && acc_ok && !*abort) {
        const int t = threadIdx.x, q = t & 3;
        const int upr = D_UNITS / ks;   // units finished per CTA
        const bf16* bias = L.bias[kv];
        const bool knorm = is_k && L.k_norm;
        for (int i = t >> 2; i < n; i += D_DEQ_THREADS / 4) {
            const int64_t ioff = s_ioff[i];
            if (ioff < 0) continue;
            // Every load of the item is issued before any of them is used (one L2
            // round trip), then the sums.
            float ssv[4];
#pragma unroll
            for (int src = 0; src < 4; ++src) ssv[src] = src < ks ? ld_l2_f32(part_ss + src * a.n_max + i) : 0.f;
            for (int ul = 0; ul < upr; ++ul) {
                const int u = rank + ul * ks;
                const int col_lo = unit_col_lo(gk, u, a.hd);
                const int head = col_lo / a.hd, seg_off = col_lo - head * a.hd;   // 32 * segment
                float4 pv[4][4];
#pragma unroll
                for (int src = 0; src < 4; ++src) {
                    if (src < ks) {
                        const float4* row = part + static_cast<int64_t>((src * D_UNITS + u) * 16) * a.n_max + i;
                        pv[src][0] = ld_l2_f4(row + static_cast<int64_t>(2 * q) * a.n_max);
                        pv[src][1] = ld_l2_f4(row + static_cast<int64_t>(2 * q + 1) * a.n_max);
                        pv[src][2] = ld_l2_f4(row + static_cast<int64_t>(8 + 2 * q) * a.n_max);
                        pv[src][3] = ld_l2_f4(row + static_cast<int64_t>(9 + 2 * q) * a.n_max);
                    } else {
#pragma unroll
                        for (int e = 0; e < 4; ++e) pv[src][e] = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
                float4 c2[4];   // {cos, sin} of the 8 pairs (K only), with the partials
                if (is_k) {
                    const float4* cs = reinterpret_cast<const float4*>(a.rope + static_cast<int64_t>(s_pos[i]) * a.half +
                                                                       seg_off + 8 * q);
#pragma unroll
                    for (int e2 = 0; e2 < 4; ++e2) c2[e2] = __ldg(cs + e2);
                }
                const float rs = 1.0f / sqrtf((ssv[0] + ssv[1] + ssv[2] + ssv[3]) * a.inv_d + a.eps);
                float lo[8], hi[8];
                sum_partials(pv, ks, rs, bias, head * a.hd + seg_off + 8 * q, a.half, lo, hi);
                if (knorm) {
                    // the head's RMS: this unit's 64 columns over the item's four
                    // threads, plus (head_dim 128) the partner unit's, summed the same way
                    float hss = 0.f;
#pragma unroll
                    for (int e = 0; e < 8; ++e) hss = fmaf(lo[e], lo[e], fmaf(hi[e], hi[e], hss));
                    if (a.hd == 128) {
                        // the partner unit's totals, one split at a time (registers)
                        float4 t4[4] = {};
#pragma unroll 1
                        for (int src = 0; src < ks; ++src) {
                            const float4* row = part + static_cast<int64_t>((src * D_UNITS + (u ^ 1)) * 16) * a.n_max + i;
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float4 v = ld_l2_f4(row + static_cast<int64_t>((e >> 1) * 8 + 2 * q + (e & 1)) * a.n_max);
                                t4[e].x += v.x;
                                t4[e].y += v.y;
                                t4[e].z += v.z;
                                t4[e].w += v.w;
                            }
                        }
                        float lo2[8] = {t4[0].x, t4[0].y, t4[0].z, t4[0].w, t4[1].x, t4[1].y, t4[1].z, t4[1].w};
                        float hi2[8] = {t4[2].x, t4[2].y, t4[2].z, t4[2].w, t4[3].x, t4[3].y, t4[3].z, t4[3].w};
                        float b[8] = {};
                        const int col2 = head * a.hd + (32 - seg_off) + 8 * q;
                        if (bias) load8_bf16(bias + col2, b);
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float x = fmaf(lo2[e], rs, b[e]);
                            hss = fmaf(x, x, hss);
                        }
                        if (bias) load8_bf16(bias + col2 + a.half, b);
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float x = fmaf(hi2[e], rs, b[e]);
                            hss = fmaf(x, x, hss);
                        }
                    }
                    const unsigned quad = 0xFu << (threadIdx.x & 28);
                    hss += __shfl_xor_sync(quad, hss, 1);
                    hss += __shfl_xor_sync(quad, hss, 2);
                    const float hs = 1.0f / sqrtf(hss / static_cast<float>(a.hd) + a.eps);
                    float g[8];
                    load8_bf16(L.k_norm + seg_off + 8 * q, g);
#pragma unroll
                    for (int e = 0; e < 8; ++e) lo[e] *= hs * g[e];
                    load8_bf16(L.k_norm + a.half + seg_off + 8 * q, g);
#pragma unroll
                    for (int e = 0; e < 8; ++e) hi[e] *= hs * g[e];
                }
                if (is_k) {
#pragma unroll
                    for (int e2 = 0; e2 < 4; ++e2) {
                        const float x1 = lo[2 * e2], x2 = hi[2 * e2];
                        const float y1 = lo[2 * e2 + 1], y2 = hi[2 * e2 + 1];
                        lo[2 * e2] = x1 * c2[e2].x - x2 * c2[e2].y;
                        hi[2 * e2] = x2 * c2[e2].x + x1 * c2[e2].y;
                        lo[2 * e2 + 1] = y1 * c2[e2].z - y2 * c2[e2].w;
                        hi[2 * e2 + 1] = y2 * c2[e2].z + y1 * c2[e2].w;
                    }
                }
                bf16* dst = (is_k ? a.kc : a.vc) + ioff + static_cast<int64_t>(head) * a.cl.s_head + seg_off + 8 * q;
                *reinterpret_cast<uint4*>(dst) = make_uint4(pack_bf16x2(lo[0], lo[1]), pack_bf16x2(lo[2], lo[3]),
                                                            pack_bf16x2(lo[4], lo[5]), pack_bf16x2(lo[6], lo[7]));
                *reinterpret_cast<uint4*>(dst + a.half) = make_uint4(pack_bf16x2(hi[0], hi[1]), pack_bf16x2(hi[2], hi[3]),
                                                                     pack_bf16x2(hi[4], hi[5]), pack_bf16x2(hi[6], hi[7]));
            }
        }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == D_MMA_WARP) tc::tmem_dealloc(tmem, D_GCOLS);
}

bool decode_eligible(const FillCall& fc) {
    const tee_fill_desc& D = *fc.desc;
    if (D.dtype != TEE_BF16 || D.wfmt != TEE_W_INT4 || D.group != D_KB) return false;
    if (fc.n_max > D_MAX_ITEMS || fc.n_layers > MAX_DECODE_LAYERS) return false;
    if (D.d % D_CH || (D.head_dim != 64 && D.head_dim != 128)) return false;
    const int kvw = D.n_kv_heads * D.head_dim;
    if (kvw % D_GCOLS) return false;
    if ((fc.ld_h * 2) % 16 || !aligned16(fc.h) || !aligned16(fc.k_cache) || !aligned16(fc.v_cache)) return false;
    const tee_cache_layout& cl = *fc.cache;
    if (cl.s_layer % 8 || cl.s_seq % 8 || cl.s_head % 8 || cl.s_pos % 8) return false;
    for (int l = 0; l < fc.n_layers; ++l) {
        const tee_fill_layer& L = fc.layers[l];
        if (L.w_map) return false;
        if (!aligned16(L.wk) || !aligned16(L.wv) || !aligned16(L.k_scale) || !aligned16(L.k_zero) ||
            !aligned16(L.v_scale) || !aligned16(L.v_zero) || !aligned16(L.gamma))
            return false;
    }
    return true;
}

// K split: the largest of 4, 2, 1 that divides d into whole chunks and keeps the
// grid within the clusters that can be resident at once.
int choose_ks(int d, int ctas_per_split, int max_clusters_4, int max_clusters_2) {
    const int sms = sm_count();
    if (d % (4 * D_CH) == 0 && ctas_per_split * 4 <= sms && ctas_per_split <= max_clusters_4) return 4;
    if (d % (2 * D_CH) == 0 && ctas_per_split * 2 <= sms && ctas_per_split <= max_clusters_2) return 2;
    return 1;
}

template <bool NARROW>
tee_status launch(const DecodeArgs& a, dim3 grid, int ks, bool early, void* ws, cudaStream_t stream) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(D_THREADS);
    cfg.dynamicSmemBytes = DLayout<NARROW>::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = early ? 2 : 1;
    const tee_status st = cuda_status(cudaLaunchKernelEx(&cfg, fill_decode_kernel<NARROW>, a, ws));
    return st != TEE_OK ? st : launch_status();   // counts the launch
}

// Clusters of ks CTAs that can be resident at once (both layouts take one CTA per SM).
int max_clusters(int ks) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(ks * 64, 1);
    cfg.blockDim = dim3(D_THREADS);
    cfg.dynamicSmemBytes = DLayout<false>::SMEM;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fill_decode_kernel<false>, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

// Workspace of the cross-CTA reduction: per cluster and rank, 64 float4 and one
// float per item row.
constexpr size_t D_PART_BUDGET = size_t(64) << 20;
size_t part_bytes(int groups_kv, int n_layers, int ks, int n_max) {
    const size_t rows = static_cast<size_t>(2 * groups_kv) * n_layers * ks * n_max;
    return round_up(rows * D_UNITS * 16 * sizeof(float4), 256) + round_up(rows * sizeof(float), 256);
}

}  // namespace

size_t fill_decode_ws_bytes(const tee_fill_desc& D, int n_layers, int n_max) {
    const int kvw = D.n_kv_heads * D.head_dim;
    if (kvw <= 0 || kvw % D_GCOLS || n_max <= 0 || n_max > D_MAX_ITEMS) return TEE_WS_HEADER_BYTES;
    for (int ks = 4; ks >= 1; ks >>= 1) {   // the largest split whose partials fit the budget
        const size_t b = part_bytes(kvw / D_GCOLS, n_layers, ks, n_max);
        if (b <= D_PART_BUDGET) return TEE_WS_HEADER_BYTES + b;
    }
    return TEE_WS_HEADER_BYTES;
}

tee_status fill_decode_run(const FillCall& fc) {
    if (!decode_eligible(fc)) return TEE_ERR_UNSUPPORTED;
    const tee_fill_desc& D = *fc.desc;
    static bool attr_set = false;
    static int mc4 = 0, mc2 = 0;
    if (!attr_set) {
        tee_status st = cuda_status(cudaFuncSetAttribute(
            fill_decode_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(DLayout<false>::SMEM)));
        if (st != TEE_OK) return st;
        st = cuda_status(cudaFuncSetAttribute(fill_decode_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              static_cast<int>(DLayout<true>::SMEM)));
        if (st != TEE_OK) return st;
        mc4 = max_clusters(4);
        mc2 = max_clusters(2);
        attr_set = true;
    }
    DecodeArgs a{};
    a.n_max = fc.n_max;
    a.n_dev = fc.n_dev;
    a.d = D.d;
    a.kvw = D.n_kv_heads * D.head_dim;
    a.hd = D.head_dim;
    a.half = D.head_dim / 2;
    a.groups_kv = a.kvw / D_GCOLS;
    a.inv_d = 1.0f / static_cast<float>(D.d);
    a.eps = D.eps;
    a.h = static_cast<const bf16*>(fc.h);
    a.ld_h = fc.ld_h;
    a.h_rows = fc.h_rows;
    a.rows = fc.rows;
    a.pos = fc.pos;
    a.pos0 = fc.pos0;
    a.seq = fc.seq;
    const PrepView pv = prep_view(fc.prep, D, fc.n_layers);
    a.hdr = pv.hdr;
    a.rope = pv.rope;
    a.kc = static_cast<bf16*>(fc.k_cache);
    a.vc = static_cast<bf16*>(fc.v_cache);
    a.cl = *fc.cache;
    for (int l = 0; l < fc.n_layers; ++l) {
        const tee_fill_layer& L = fc.layers[l];
        a.l[l] = DecodeLayer{{static_cast<const uint8_t*>(L.wk), static_cast<const uint8_t*>(L.wv)},
                             {static_cast<const __half*>(L.k_scale), static_cast<const __half*>(L.v_scale)},
                             {static_cast<const __half*>(L.k_zero), static_cast<const __half*>(L.v_zero)},
                             static_cast<const bf16*>(L.gamma),
                             {static_cast<const bf16*>(L.k_bias), static_cast<const bf16*>(L.v_bias)},
                             static_cast<const bf16*>(L.k_norm), L.cache_layer, L.writes};
    }
    const int splits = 2 * a.groups_kv * fc.n_layers;   // (group, layer) pairs
    a.ks = choose_ks(D.d, splits, mc4, mc2);
    while (a.ks > 1 && TEE_WS_HEADER_BYTES + part_bytes(a.groups_kv, fc.n_layers, a.ks, fc.n_max) > fc.ws_bytes)
        a.ks >>= 1;   // a smaller split needs smaller partials
    if (TEE_WS_HEADER_BYTES + part_bytes(a.groups_kv, fc.n_layers, a.ks, fc.n_max) > fc.ws_bytes ||
        D.d / a.ks > D_MAX_KC)
        return TEE_ERR_UNSUPPORTED;
    {
        char* p = static_cast<char*>(fc.ws) + TEE_WS_HEADER_BYTES;
        const size_t rows = static_cast<size_t>(2 * a.groups_kv) * fc.n_layers * a.ks * fc.n_max;
        a.part = reinterpret_cast<float4*>(p);
        a.part_ss = reinterpret_cast<float*>(p + round_up(rows * D_UNITS * 16 * sizeof(float4), 256));
    }
    const dim3 grid(2 * a.groups_kv * a.ks, fc.n_layers);
    // An early launch parks the grid's CTAs on their SMs until the previous kernel
    // completes: only when the grid leaves SMs free for that kernel to finish on.
    const bool early = (D.flags & TEE_FILL_EARLY_WEIGHTS) && static_cast<int>(grid.x * grid.y) + 4 <= sm_count();
    return fc.n_max <= DLayout<true>::ITEMS ? launch<true>(a, grid, a.ks, early, fc.ws, fc.stream)
                                            : launch<false>(a, grid, a.ks, early, fc.ws, fc.stream);
}

}  // namespace tee
