// Decode path of the KV fill: up to 128 items (decode tokens that exit), int4
// group-64 weights (River-LLM's W4A16 exit layers), identity map (the
// "State Propagation" / identity-fill input).
//
// Work split. The K and V projections of one filled layer are cut into groups
// of 256 output columns, and the reduction dimension d into KS equal ranges.
// One cluster of KS CTAs per (group, layer): CTA r computes, on tcgen05,
//   P_r[item][c] = sum_{k in range r} (h[row(item)][k] g_j[k]) * W[k][c],
//   W[k][c] = (q - zero) * scale     (M = 128 item rows, N = 256, K = d / KS)
// and the partial sums of h^2 over its range; the CTAs then add their partials
// through distributed shared memory. A group is four units of 64 columns, each
// unit the two 32-wide halves [i, i+32) and [i+hd/2, i+hd/2+32) of one head,
// so that RoPE pairs stay inside a unit; unit u is finished by the CTA of rank
// u % KS: sum of the KS partials, 1/rms over the whole d, RoPE, bf16 store
// into the backbone's cache slot.
//
// Warp roles in a CTA (mbarriers between roles):
//   warps 0-7   stream the CTA's int4 codes and fp16 scales/zeros (cp.async, 256-k
//               chunks, two in flight) and dequantise each 64-k block into a ring
//               of bf16 B operands (256 rows of 128 bytes, 128-byte swizzle):
//               W[k][c] = (q - z) s, in packed bf16x2 arithmetic;
//   warp 8      issues tcgen05.mma (N = 256) into a 256-column TMEM accumulator;
//   warps 9-12  gather the items' h rows of each 64-k block into a ring of A
//               operands (cp.async, 128-byte swizzle), after asking L2 for the
//               rows' slices at the start. Once a thread's pieces of a block have
//               landed it adds their squares into per-item sums of h^2 and scales
//               them by the RMSNorm gain g_j in place (A = h * g_j), then releases
//               the block; they also fetch positions and cache slots.
// After the last MMA, in rounds of 64 item rows: warps 0-7 copy the accumulator
// rows (thread = item row) into shared memory per unit, with the row's partial
// sum of h^2 in the padding; a cluster barrier; one thread sends each unit's
// rows to its finishing CTA with a bulk shared::cluster copy that completes on
// the receiver's mbarrier; the receivers add the partials and finish; a
// cluster barrier closes the round.
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
constexpr int D_RB = 2;              // B operand slots (dequantised weights)
constexpr int D_RC = 2;              // code chunks in flight
constexpr int D_MAX_ITEMS = 128;
constexpr int D_DEQ_WARPS = 8, D_MMA_WARP = 8, D_CP_WARP0 = 9, D_CP_WARPS = 4;
constexpr int D_DEQ_THREADS = D_DEQ_WARPS * 32;
constexpr int D_CP_THREADS = D_CP_WARPS * 32;
constexpr int D_ITEMS_PER_CP = D_MAX_ITEMS * 8 / D_CP_THREADS;   // 16-byte pieces per thread and block
constexpr int D_THREADS = (D_CP_WARP0 + D_CP_WARPS) * 32;
constexpr int D_MAX_KC = 2048;       // largest k range of one CTA (its g_j slice sits in shared memory)
// A slot is refilled D_RA - D_LAG - 1 iterations after its release: slack for the
// MMA round trip (an mbarrier hand-off costs ~0.1 us).
static_assert(D_LAG + 2 < D_RA, "the A ring needs slack beyond the blocks in flight");

constexpr uint32_t A_SLOT = 128 * 128;                  // 16 KB: 128 item rows x 64 k
constexpr uint32_t B_SLOT = D_GCOLS * 128;              // 32 KB: 256 columns x 64 k
constexpr uint32_t CH_CODES = (D_CH / 2) * D_GCOLS;     // 32 KB: 128 packed rows x 256 columns
constexpr uint32_t CH_SZ = (D_CH / D_KB) * D_GCOLS * 4; // 4 KB: scale[256], zero[256] (fp16) per group
constexpr uint32_t CH_BYTES = CH_CODES + CH_SZ;
constexpr uint32_t OFF_A = 0;
constexpr uint32_t OFF_B = OFF_A + D_RA * A_SLOT;
constexpr uint32_t OFF_C = OFF_B + D_RB * B_SLOT;
constexpr uint32_t OFF_G = OFF_C + D_RC * CH_BYTES;               // g_j over this CTA's k range (bf16)
constexpr uint32_t OFF_SMALL = OFF_G + D_MAX_KC * 2;
constexpr uint32_t SMALL_BYTES = (2 * D_RA + 2 * D_RB + 3) * 8 + D_MAX_ITEMS * (8 + 4 + 4) + 16;
constexpr size_t D_SMEM = 1024 + OFF_SMALL + SMALL_BYTES;
// After the main loop the operand and code rings hold, per round of 64 item rows, this CTA's
// partials [unit][row][P_LD floats] (64 unit columns, then the row's partial sum of
// h^2, padding) and the partials received for the units it finishes
// [slot = source rank * units per CTA + owned unit][row][P_LD floats].
constexpr int P_LD = 68;
constexpr int P_ROWS = 64;
constexpr uint32_t P_ROW_BYTES = P_LD * 4;
constexpr uint32_t P_TILE = P_ROWS * P_ROW_BYTES;
constexpr uint32_t OFF_STG = 0;
constexpr uint32_t OFF_RCV = OFF_STG + D_UNITS * P_TILE;
static_assert(OFF_RCV + D_UNITS * P_TILE <= OFF_G, "the partials fit in the operand and code rings");
static_assert(D_SMEM <= 232448, "decode fill shared memory");
static_assert(OFF_B % 1024 == 0 && OFF_C % 16 == 0 && OFF_G % 16 == 0 && OFF_SMALL % 8 == 0, "alignment");

struct DecodeLayer {
    const uint8_t* codes[2];   // wk, wv
    const __half* scale[2];
    const __half* zero[2];
    const bf16* gamma;
    int cache_layer;
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
// (q - 8) s + (8 - z) s = (q - z) s, rounded once. wl / wh: the packed word and the
// word shifted right by 4; sel picks byte b of each into bytes 0 and 2.
__device__ __forceinline__ uint32_t deq_pair(uint32_t wl, uint32_t wh, uint32_t sel, __nv_bfloat162 s2,
                                             __nv_bfloat162 zs2) {
    const uint32_t x = (__byte_perm(wl, wh, sel) & 0x000F000Fu) | 0x43004300u;
    __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&x);
    v = __hfma2(__hsub2(v, __floats2bfloat162_rn(136.0f, 136.0f)), s2, zs2);
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
__device__ __forceinline__ uint32_t map_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
// Bulk copy of bytes from this CTA's shared memory to a cluster peer's, completing
// on the peer's mbarrier (both given as shared::cluster addresses).
__device__ __forceinline__ void bulk_to_peer(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t mbar) {
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "r"(src), "r"(bytes), "r"(mbar)
                 : "memory");
}

// First column of unit u's low and high halves within the K (or V) projection.
__device__ __forceinline__ int unit_col_lo(int gk, int u, int hd) {
    const int uph = hd / 64;   // units per head
    return (D_GCOLS * gk / hd + u / uph) * hd + 32 * (u % uph);
}

__global__ void __launch_bounds__(D_THREADS, 1)
fill_decode_kernel(const __grid_constant__ DecodeArgs a, void* ws) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* a_full = reinterpret_cast<uint64_t*>(smem + OFF_SMALL);
    uint64_t* a_empty = a_full + D_RA;
    uint64_t* b_full = a_empty + D_RA;
    uint64_t* b_empty = b_full + D_RB;
    uint64_t* acc_full = b_empty + D_RB;
    uint64_t* ss_ready = acc_full + 1;
    uint64_t* recv_full = ss_ready + 1;
    int64_t* s_ioff = reinterpret_cast<int64_t*>(recv_full + 1);   // item part of the cache offset, or -1
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
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kc = a.d / ks, k0 = rank * kc;     // this CTA's k range
    const int nkb = kc / D_KB, nch = kc / D_CH;
    const int n = min(item_count(a.n_max, a.n_dev), D_MAX_ITEMS);
    const bool reporter = blockIdx.x == 0 && li == 0;   // one CTA records bad rows / positions

    if (threadIdx.x == 0) {
        for (int s = 0; s < D_RA; ++s) {
            tc::mbar_init(&a_full[s], D_CP_WARPS);
            tc::mbar_init(&a_empty[s], 1);                // MMA commit
        }
        for (int s = 0; s < D_RB; ++s) {
            tc::mbar_init(&b_full[s], D_DEQ_WARPS);
            tc::mbar_init(&b_empty[s], 1);
        }
        tc::mbar_init(acc_full, 1);
        tc::mbar_init(ss_ready, D_CP_WARPS);
        tc::mbar_init(recv_full, 1);
        *abort = 0;
        tc::fence_barrier_init();
    }
    // Chunk c of the CTA's codes / scales / zeros into ring slot c % D_RC. Staged
    // column order: unit u's low half, then its high half (64 u .. 64 u + 63).
    auto load_chunk = [&](int c) {
        uint8_t* base = smem + OFF_C + (c % D_RC) * CH_BYTES;
        const int kg = k0 + c * D_CH;             // first k of the chunk
        for (int v = threadIdx.x; v < (D_CH / 2) * 16; v += D_DEQ_THREADS) {
            const int r = v >> 4, p = v & 15, u = p >> 2, part = p & 3;
            const int col = unit_col_lo(gk, u, a.hd) + (part >= 2 ? a.half : 0) + (part & 1) * 16;
            cp_async16(base + r * D_GCOLS + p * 16, L.codes[kv] + static_cast<int64_t>(kg / 2 + r) * a.kvw + col);
        }
        for (int v = threadIdx.x; v < D_BPC * 64; v += D_DEQ_THREADS) {
            // group g, scale or zero, unit u, half: 32 fp16 = 4 pieces
            const int g = v >> 6, which = (v >> 5) & 1, p = v & 31, u = p >> 3, hp = (p >> 2) & 1, q = p & 3;
            const int col = unit_col_lo(gk, u, a.hd) + (hp ? a.half : 0) + q * 8;
            const __half* src = (which ? L.zero[kv] : L.scale[kv]) + static_cast<int64_t>(kg / D_KB + g) * a.kvw + col;
            cp_async16(base + CH_CODES + g * (D_GCOLS * 4) + which * (D_GCOLS * 2) + (u * 64 + hp * 32 + q * 8) * 2, src);
        }
    };
    if (warp < D_DEQ_WARPS) {
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
            const uint8_t* base = smem + OFF_C + (c % D_RC) * CH_BYTES;
            for (int b = 0; b < D_BPC && ok; ++b) {
                const int kb = c * D_BPC + b, s = kb % D_RB;
                if (kb >= D_RB && !warp_wait(&b_empty[s], ((kb / D_RB) - 1) & 1, abort, ws, 51)) {
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
                uint8_t* bslot = smem + OFF_B + s * B_SLOT;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const __nv_bfloat162 s2 = __floats2bfloat162_rn(sc[j], sc[j]);
                    const float zs = (8.0f - zr[j]) * sc[j];
                    const __nv_bfloat162 zs2 = __floats2bfloat162_rn(zs, zs);
                    const uint32_t sel = (j | (j << 4) | ((j + 4) << 8) | ((j + 4) << 12));
                    uint32_t o[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) o[i] = deq_pair(w[i], wh[i], sel, s2, zs2);   // k 16 kq + 2i, +1
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
                const int sa = kb % D_RA, sb = kb % D_RB;
                if (!tc::mbar_wait(&a_full[sa], (kb / D_RA) & 1, abort, ws, 53)) break;
                if (!tc::mbar_wait(&b_full[sb], (kb / D_RB) & 1, abort, ws, 54)) break;
                tc::tc_fence_after();
                const uint64_t ad = tc::smem_desc_sw128(tc::smem_u32(smem + OFF_A + sa * A_SLOT));
                const uint64_t bd = tc::smem_desc_sw128(tc::smem_u32(smem + OFF_B + sb * B_SLOT));
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
        // This CTA's slice of g_j (landed before the first release, see below).
        for (int v = ct; v < kc / 8; v += D_CP_THREADS) cp_async16(smem + OFF_G + v * 16, L.gamma + k0 + v * 8);
        cp_async_commit();   // the oldest group
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
        const bf16* src[D_ITEMS_PER_CP];
#pragma unroll
        for (int m = 0; m < D_ITEMS_PER_CP; ++m) {
            const int i = ib + 16 * m;
            const int r = i < n ? (a.rows ? a.rows[i] : i) : -1;
            src[m] = (r >= 0 && r < a.h_rows) ? a.h + static_cast<int64_t>(r) * a.ld_h + k0 + j * 8 : nullptr;
        }
        auto issue = [&](int kb) {
            uint8_t* slot = smem + OFF_A + (kb % D_RA) * A_SLOT;
#pragma unroll
            for (int m = 0; m < D_ITEMS_PER_CP; ++m) {
                const int i = ib + 16 * m;
                if (src[m]) cp_async16(slot + i * 128 + ((j ^ (i & 7)) << 4), src[m] + kb * D_KB);
            }
        };
        float ss[D_ITEMS_PER_CP];
#pragma unroll
        for (int m = 0; m < D_ITEMS_PER_CP; ++m) ss[m] = 0.f;
        // Block kb's pieces of this thread have landed: add their squares, scale them
        // by g_j (bf16 x bf16 -> bf16, one rounding), order them for the tensor core,
        // and release the block once the whole warp is done.
        auto release = [&](int kb) {
            uint8_t* slot = smem + OFF_A + (kb % D_RA) * A_SLOT;
            const uint4 gp = *reinterpret_cast<const uint4*>(smem + OFF_G + (kb * D_KB + 8 * j) * 2);
            const __nv_bfloat162* gv = reinterpret_cast<const __nv_bfloat162*>(&gp);
#pragma unroll
            for (int m = 0; m < D_ITEMS_PER_CP; ++m) {
                if (!src[m]) continue;
                const int i = ib + 16 * m;
                uint4* pp = reinterpret_cast<uint4*>(slot + i * 128 + ((j ^ (i & 7)) << 4));
                uint4 x = *pp;
                ss[m] = sumsq8(x, ss[m]);
                __nv_bfloat162* xv = reinterpret_cast<__nv_bfloat162*>(&x);
#pragma unroll
                for (int e = 0; e < 4; ++e) xv[e] = __hmul2(xv[e], gv[e]);
                *pp = x;
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&a_full[kb % D_RA]);
        };
        // The g_j slice comes from every copier: they meet once, after their first wait.
        auto g_ready = [&]() { asm volatile("bar.sync 2, %0;" ::"n"(D_CP_THREADS) : "memory"); };
        bool ok = true;
        int waited = 0;
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
                if (!waited) {
                    g_ready();
                    waited = 1;
                }
                release(kb - D_LAG);
            }
        }
        cp_async_wait<0>();
        if (!waited) g_ready();   // every copier reaches the meeting exactly once
        if (ok)
            for (int b = max(0, nkb - D_LAG); b < nkb; ++b) release(b);
        // Per-item totals: the eight threads of an item are consecutive lanes.
#pragma unroll
        for (int m = 0; m < D_ITEMS_PER_CP; ++m) {
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

    // ---- the reduction across the cluster, in rounds of 64 item rows.
    // Accumulator column cg + 64 j holds staged column 4 cg + j, i.e. unit cg / 16,
    // unit column 4 (cg % 16) + j.
    bool acc_ok = true;
    if (warp < D_DEQ_WARPS) {
        acc_ok = warp_wait(acc_full, 0, abort, ws, 56);
        acc_ok = warp_wait(ss_ready, 0, abort, ws, 57) && acc_ok;   // s_ss, s_ioff, s_pos
        tc::tc_fence_after();
    }
    const int upr = D_UNITS / ks;   // units finished per CTA
    const uint32_t stg_s = tc::smem_u32(smem + OFF_STG), rcv_s = tc::smem_u32(smem + OFF_RCV);
    const float* stg = reinterpret_cast<const float*>(smem + OFF_STG);
    const float* rcv = reinterpret_cast<const float*>(smem + OFF_RCV);
    const int rounds = (n + P_ROWS - 1) / P_ROWS;
    for (int round = 0; round < rounds; ++round) {
        const int r0 = round * P_ROWS, nr = min(P_ROWS, n - r0);
        if (threadIdx.x == 0 && ks > 1)
            tc::mbar_arrive_expect_tx(recv_full, static_cast<uint32_t>(upr * (ks - 1) * nr) * P_ROW_BYTES);
        // Rows r0 .. r0 + 63 sit in TMEM lane quarters 2 round, 2 round + 1: warps w with
        // w % 4 in those quarters read them, units 0-1 (w < 4) or 2-3 (w >= 4).
        if (warp < D_DEQ_WARPS && (warp & 3) / 2 == round) {
            const int r = (warp & 3) * 32 + lane, rl = r - r0;
            const uint32_t tb = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
#pragma unroll 1
            for (int u = 2 * (warp >> 2); u < 2 * (warp >> 2) + 2; ++u) {
                float v[4][16];
#pragma unroll
                for (int j = 0; j < 4; ++j) tc::tmem_ld16(tb + 16 * u + 64 * j, v[j]);   // warp-wide
                if (rl < nr) {
                    float* row = reinterpret_cast<float*>(smem + OFF_STG + u * P_TILE + rl * P_ROW_BYTES);
#pragma unroll
                    for (int m = 0; m < 16; ++m)
                        *reinterpret_cast<float4*>(row + 4 * m) = make_float4(v[0][m], v[1][m], v[2][m], v[3][m]);
                    row[64] = s_ss[r];
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // read next by the bulk copies
        }
        tc::tc_fence_before();
        __syncthreads();
        cluster_sync();   // partials staged everywhere; every receiver's rings are free
        tc::tc_fence_after();
        if (threadIdx.x == 0)
            for (int u = 0; u < D_UNITS; ++u) {
                const int owner = u % ks;
                if (owner == rank) continue;
                const int slot = rank * upr + u / ks;
                bulk_to_peer(map_rank(rcv_s + slot * P_TILE, owner), stg_s + u * P_TILE,
                             static_cast<uint32_t>(nr) * P_ROW_BYTES, map_rank(tc::smem_u32(recv_full), owner));
            }
        // ---- finish the units of this rank: warps 0-7, thread = (item, 8 column pairs).
        if (warp < D_DEQ_WARPS) {
            const bool got = ks == 1 || warp_wait(recv_full, round & 1, abort, ws, 58);
            const int t = threadIdx.x, q = t & 3, il = t >> 2, i = r0 + il;
            if (got && acc_ok && !*abort && il < nr && s_ioff[i] >= 0) {
                const int64_t ioff = s_ioff[i];
                for (int ul = 0; ul < upr; ++ul) {
                    const int u = rank + ul * ks;
                    const int col_lo = unit_col_lo(gk, u, a.hd);
                    const int head = col_lo / a.hd, seg_off = col_lo - head * a.hd;   // 32 * segment
                    float lo[8], hi[8], ss = 0.f;
#pragma unroll
                    for (int e = 0; e < 8; ++e) lo[e] = hi[e] = 0.f;
                    for (int src = 0; src < ks; ++src) {
                        const float* row = (src == rank ? stg + (u * P_ROWS + il) * P_LD
                                                        : rcv + ((src * upr + ul) * P_ROWS + il) * P_LD);
                        const float4 l0 = *reinterpret_cast<const float4*>(row + 8 * q);
                        const float4 l1 = *reinterpret_cast<const float4*>(row + 8 * q + 4);
                        const float4 h0 = *reinterpret_cast<const float4*>(row + 32 + 8 * q);
                        const float4 h1 = *reinterpret_cast<const float4*>(row + 32 + 8 * q + 4);
                        lo[0] += l0.x; lo[1] += l0.y; lo[2] += l0.z; lo[3] += l0.w;
                        lo[4] += l1.x; lo[5] += l1.y; lo[6] += l1.z; lo[7] += l1.w;
                        hi[0] += h0.x; hi[1] += h0.y; hi[2] += h0.z; hi[3] += h0.w;
                        hi[4] += h1.x; hi[5] += h1.y; hi[6] += h1.z; hi[7] += h1.w;
                        ss += row[64];
                    }
                    const float rs = 1.0f / sqrtf(ss * a.inv_d + a.eps);
                    if (is_k) {
                        const float4* cs = reinterpret_cast<const float4*>(
                            a.rope + static_cast<int64_t>(s_pos[i]) * a.half + seg_off + 8 * q);
#pragma unroll
                        for (int e2 = 0; e2 < 4; ++e2) {
                            const float4 c2 = __ldg(cs + e2);   // {cos, sin} of two pairs
                            const float x1 = lo[2 * e2] * rs, x2 = hi[2 * e2] * rs;
                            const float y1 = lo[2 * e2 + 1] * rs, y2 = hi[2 * e2 + 1] * rs;
                            lo[2 * e2] = x1 * c2.x - x2 * c2.y;
                            hi[2 * e2] = x2 * c2.x + x1 * c2.y;
                            lo[2 * e2 + 1] = y1 * c2.z - y2 * c2.w;
                            hi[2 * e2 + 1] = y2 * c2.z + y1 * c2.w;
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            lo[e] *= rs;
                            hi[e] *= rs;
                        }
                    }
                    bf16* dst = (is_k ? a.kc : a.vc) + ioff + static_cast<int64_t>(head) * a.cl.s_head + seg_off + 8 * q;
                    *reinterpret_cast<uint4*>(dst) = make_uint4(pack_bf16x2(lo[0], lo[1]), pack_bf16x2(lo[2], lo[3]),
                                                                pack_bf16x2(lo[4], lo[5]), pack_bf16x2(lo[6], lo[7]));
                    *reinterpret_cast<uint4*>(dst + a.half) =
                        make_uint4(pack_bf16x2(hi[0], hi[1]), pack_bf16x2(hi[2], hi[3]), pack_bf16x2(hi[4], hi[5]),
                                   pack_bf16x2(hi[6], hi[7]));
                }
            }
        }
        cluster_sync();   // the round's copies have landed and been read: buffers reusable, peers may exit
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

tee_status launch(const DecodeArgs& a, dim3 grid, int ks, void* ws, cudaStream_t stream) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(D_THREADS);
    cfg.dynamicSmemBytes = D_SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const tee_status st = cuda_status(cudaLaunchKernelEx(&cfg, fill_decode_kernel, a, ws));
    return st != TEE_OK ? st : launch_status();   // counts the launch
}

int max_clusters(int ks) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(ks * 64, 1);
    cfg.blockDim = dim3(D_THREADS);
    cfg.dynamicSmemBytes = D_SMEM;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fill_decode_kernel, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace

size_t fill_decode_ws_bytes(const tee_fill_desc& D, int n_layers, int n_max) {
    (void)D;
    (void)n_layers;
    (void)n_max;
    return TEE_WS_HEADER_BYTES;
}

tee_status fill_decode_run(const FillCall& fc) {
    if (!decode_eligible(fc)) return TEE_ERR_UNSUPPORTED;
    const tee_fill_desc& D = *fc.desc;
    static bool attr_set = false;
    static int mc4 = 0, mc2 = 0;
    if (!attr_set) {
        tee_status st = cuda_status(cudaFuncSetAttribute(fill_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                         static_cast<int>(D_SMEM)));
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
                             static_cast<const bf16*>(L.gamma), L.cache_layer};
    }
    const int splits = 2 * a.groups_kv * fc.n_layers;   // (group, layer) pairs
    a.ks = choose_ks(D.d, splits, mc4, mc2);
    if (D.d / a.ks > D_MAX_KC) return TEE_ERR_UNSUPPORTED;
    return launch(a, dim3(2 * a.groups_kv * a.ks, fc.n_layers), a.ks, fc.ws, fc.stream);
}

}  // namespace tee
