// Decode path of the KV fill: up to 128 items (decode tokens that exit), int4
// group-64 weights (River-LLM's W4A16 exit layers), identity map (the
// "State Propagation" / identity-fill input).
//
// Work split. The K and V projections of every filled layer are cut into
// tiles of 128 output columns, and the reduction dimension d into KS equal
// ranges. One cluster of KS CTAs per (tile, layer); CTA r computes, on
// tcgen05, the partial
//   P_r[c][item] = sum_{k in range r} W'[k][c] h[row(item)][k],
//   W'[k][c] = (q - z) s g_j[k]   (the RMSNorm gain folded into the weights)
// with the weights as the MMA's A operand (M = the tile's 128 columns) held in
// tensor memory and the items' rows as the B operand (N = items, rounded up
// to 16) in shared memory, and the partial sums of h^2 over its range. The
// CTAs of a cluster then add their partials through distributed shared
// memory; CTA r finishes items [r N/KS, (r+1) N/KS): 1/rms over the whole d,
// bias, per-head K norm, RoPE on K, bf16 store into the backbone's slot.
//
// Prepared weights (tee_kv_fill_prepare): per (layer, K|V, tile, 64-k block)
// one 4608-byte record -- the tile's 128 columns x 64 codes as two halves of
// [128 columns][16 bytes] (column c's 32 codes of the half; in each 4-byte
// word of 8 codes, nibbles p and p + 4 hold k = 2p and 2p + 1 of the word),
// then [128 columns] {bf16 s, bf16 (8 - z) s}. A CTA's blocks are one
// contiguous run that a few bulk copies bring in at once.
//
// Warp roles in a CTA (mbarriers between roles):
//   warps 0-15  dequantise: warp w takes TMEM lane quarter w % 4 (thread =
//               tile column 32 (w % 4) + lane) and, of each chunk of four
//               blocks, block w / 4. A block of 64 codes becomes 32 bf16 pairs
//               (W' = ((q - 8) s + (8 - z) s) g_j in bf16x2 arithmetic) stored
//               with one tcgen05.st into a ring of A slots in tensor memory;
//   warp 16     allocates tensor memory and issues tcgen05.mma (A from TMEM,
//               B = the items' h block) into the accumulator;
//   warp 17     streams the CTA's prepared weights (bulk copies of four
//               blocks into a ring of chunk slots) and its slice of g_j;
//   warps 18-21 add the squares of the items' h rows to per-item sums of
//               h^2 and fetch positions and cache slots; past the first RH
//               blocks (a long k range) they also refill the B ring.
// The items' h rows of the first RH blocks (the B operands, 128-byte swizzle)
// are requested at the start: when the items are consecutive rows of h (the
// compacted batch) by warp 17 with one three-dimensional TMA copy (rows x 64-k
// blocks), otherwise by warps 0-15 and 18-21 together with cp.async (the copy
// rate per SM grows with the number of warps issuing).
// After the last MMA warps 0-15 move the accumulator (thread = column, a
// quarter of the items per warp) to a shared [item][column] fp32 tile; one
// cluster barrier; warps 0-15 of each CTA add the KS tiles of the items it
// finishes (the peers' through distributed shared memory) and store; a second
// cluster barrier keeps every tile alive until all peers have read it.
#include "fill.cuh"
#include "tc.cuh"

namespace tee {

namespace {

using bf16 = __nv_bfloat16;

constexpr int T_COLS = 128;                 // output columns per tile (MMA M, TMEM lanes)
constexpr int KB = 64;                      // k per block (one int4 group)
constexpr int CHB = 4;                      // blocks per weight chunk
constexpr uint32_t BLK_BYTES = 4608;        // prepared block record
constexpr uint32_t CODE_HALF = 2048;        // [128 columns][16 bytes]
constexpr uint32_t SC_OFF = 4096;           // [128 columns] {bf16 s, bf16 (8 - z) s}
constexpr uint32_t CHUNK_BYTES = CHB * BLK_BYTES;
constexpr int RW = 4;                       // weight chunk slots
constexpr int RA = 2 * CHB;                 // TMEM A slots (dequantised blocks): two chunks
constexpr int RAC = RA / CHB;               // chunk slots of the A ring
constexpr int ACC_COLS = 128;               // TMEM columns of the accumulator (items)
constexpr uint32_t TMEM_COLS = 512;
static_assert(ACC_COLS + 32 * RA <= static_cast<int>(TMEM_COLS), "tensor memory budget");
constexpr int DEQ_WARPS = 16, MMA_WARP = 16, LD_WARP = 17, CP_WARP0 = 18, CP_WARPS = 4;
constexpr int DEQ_THREADS = DEQ_WARPS * 32;
constexpr int CP_THREADS = CP_WARPS * 32;
constexpr int H_WARPS = DEQ_WARPS + CP_WARPS;   // warps that request the first h blocks
constexpr int THREADS = (CP_WARP0 + CP_WARPS) * 32;
constexpr int MAX_ITEMS = 128;
constexpr int MAX_NBC = 64;                 // 64-k blocks of one CTA at most (its g_j slice in shared memory)
constexpr int P_LD = T_COLS + 4;            // floats per row of the epilogue tile (bank spread)
static_assert(DEQ_WARPS == 4 * CHB, "one block of each chunk per dequantising warp of a lane quarter");

// Shared-memory layout. Up to 64 items ("narrow") the B slots hold 64 rows, up
// to 128 items 128 rows. The epilogue's [item][column] fp32 tile reuses the B
// ring once the last MMA has completed.
template <bool NARROW>
struct DLayout {
    static constexpr int ITEMS = NARROW ? 64 : 128;
    static constexpr int RH = NARROW ? 16 : 8;            // B slots (h blocks)
    static constexpr uint32_t H_SLOT = ITEMS * 128;       // item rows x 64 k (bf16)
    static constexpr uint32_t OFF_H = 0;
    static constexpr uint32_t OFF_W = OFF_H + RH * H_SLOT;
    static constexpr uint32_t OFF_G = OFF_W + RW * CHUNK_BYTES;    // g_j over the CTA's k range (bf16)
    static constexpr uint32_t OFF_SMALL = OFF_G + MAX_NBC * KB * 2;
    static constexpr int N_BARS = 2 * RH + 2 * RW + 2 * RAC + 6;
    static constexpr uint32_t SMALL_BYTES = N_BARS * 8 + MAX_ITEMS * (8 + 4 + 4) + 16;
    static constexpr size_t SMEM = 1024 + OFF_SMALL + SMALL_BYTES;
    static constexpr int IPC = ITEMS * 8 / CP_THREADS;    // 16-byte h pieces per gathering thread and block
    static constexpr int IPW = ITEMS / 4;                 // accumulator columns (items) per dequantising warp
    static_assert(static_cast<uint32_t>(ITEMS * P_LD * 4) <= RH * H_SLOT, "epilogue tile fits the B ring");
    static_assert(SMEM <= 232448, "decode fill shared memory");
    static_assert(H_SLOT % 1024 == 0 && OFF_W % 16 == 0 && OFF_SMALL % 8 == 0, "alignment");
};

struct DecodeLayer {
    const uint8_t* w;      // this layer's prepared records: [K|V][tile][block]
    const bf16* gamma;
    const bf16* bias[2];   // k_bias, v_bias (nullable)
    const bf16* k_norm;    // per-head K norm weight (nullable)
    int cache_layer;
    int writes;            // 0, TEE_FILL_WRITE_K or TEE_FILL_WRITE_V
};
constexpr int MAX_DECODE_LAYERS = 64;
struct DecodeArgs {
    DecodeLayer l[MAX_DECODE_LAYERS];
    int n_max, d, kvw, hd, half, tpk, nb, ks;   // tpk: tiles per K (or V); nb: 64-k blocks in d
    int h_tma;                                  // tm_h describes h (rows x 64-k blocks, box: items x pre blocks)
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
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(tc::smem_u32(dst)), "l"(src), "r"(bytes), "r"(tc::smem_u32(bar))
                 : "memory");
}
// Lane 0 waits for the phase, the warp follows: every lane sees the same outcome,
// so a timed-out wait cannot split a warp at a later __syncwarp or named barrier.
// Every lane tests the phase (no lane waits alone while the others park at a
// shuffle: that costs microseconds). Bounded: after tc::WAIT_LIMIT_NS, or once
// another role has raised *abort, the warp records the fault (lane 0) and
// returns false, all lanes alike.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort, void* ws, int where) {
    if (__all_sync(0xffffffffu, tc::mbar_test_wait(bar, parity))) return true;
    const uint64_t t0 = tc::globaltimer();
    for (uint32_t i = 0;; ++i) {
        if (__all_sync(0xffffffffu, tc::mbar_test_wait(bar, parity))) return true;
        if ((i & 63) == 63) {
            const int stop = __shfl_sync(0xffffffffu, (*abort != 0) ? 1 : (tc::globaltimer() - t0 > tc::WAIT_LIMIT_NS ? 2 : 0), 0);
            if (stop) {
                if (stop == 2 && (threadIdx.x & 31) == 0) {
                    *abort = 1;
                    record_fault(ws, TEE_DEVERR_TIMEOUT, where);
                }
                return false;
            }
        }
    }
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
// The four k-pairs of one prepared code word: pair p = (k 2p, k 2p + 1) of the
// word sits in nibbles p and p + 4, so (w >> 4p) & 0x000F000F | 0x43004300 is the
// exact bf16 pair 128 + q; subtracting 136 leaves q - 8 exactly, one bf16x2 fma
// gives (q - 8) s + (8 - z) s = (q - z) s, rounded once, and one bf16x2 multiply
// by the pair's RMSNorm gains (g_j[k], g_j[k + 1]) rounds again.
__device__ __forceinline__ void deq_word(uint32_t w, __nv_bfloat162 s2, __nv_bfloat162 c2, uint4 g, uint32_t* o) {
    const __nv_bfloat162 off = __floats2bfloat162_rn(136.0f, 136.0f);
    const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const uint32_t x = ((w >> (4 * p)) & 0x000F000Fu) | 0x43004300u;
        __nv_bfloat162 v = __hfma2(__hsub2(*reinterpret_cast<const __nv_bfloat162*>(&x), off), s2, c2);
        v = __hmul2(v, *reinterpret_cast<const __nv_bfloat162*>(&gw[p]));
        o[p] = *reinterpret_cast<const uint32_t*>(&v);
    }
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
        "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
        "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// D[tmem] (+)= A[tmem] * B[smem]^T: kind::f16 with A (M x 16 bf16) read from
// tensor memory (row m in lane m, k pairs packed in 32-bit columns).
__device__ __forceinline__ void umma_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n"
        "}\n" ::"r"(tmem_d),
        "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t peer_addr(const void* local, int rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(tc::smem_u32(local)), "r"(rank));
    return r;
}
__device__ __forceinline__ float4 ld_peer_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ float ld_peer_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void load8_bf16(const bf16* p, float (&v)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    unpack_bf16x2(u.x, v[0], v[1]);
    unpack_bf16x2(u.y, v[2], v[3]);
    unpack_bf16x2(u.z, v[4], v[5]);
    unpack_bf16x2(u.w, v[6], v[7]);
}

// True when the items' rows are h rows r0, r0 + 1, ... (every lane of the warp
// agrees): then one TMA copy brings all of them.
__device__ __forceinline__ bool rows_contiguous(const DecodeArgs& a, int n, int lane, int& r0) {
    r0 = (a.rows && n > 0) ? a.rows[0] : 0;
    bool ok = r0 >= 0 && r0 + n <= a.h_rows;
    if (a.rows)
        for (int i = lane; i < n; i += 32) ok = ok && a.rows[i] == r0 + i;
    return __all_sync(0xffffffffu, ok);
}

template <bool NARROW>
__global__ void __launch_bounds__(THREADS, 1)
fill_decode_kernel(const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ DecodeArgs a, void* ws) {
    using Lay = DLayout<NARROW>;
    allow_dependents();   // a dependent launched after the fill waits for it before any access
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* h_full = reinterpret_cast<uint64_t*>(smem + Lay::OFF_SMALL);   // ring blocks past the first RH
    uint64_t* h_empty = h_full + Lay::RH;
    uint64_t* w_full = h_empty + Lay::RH;
    uint64_t* w_empty = w_full + RW;
    uint64_t* a_full = w_empty + RW;                            // per chunk slot of the A ring
    uint64_t* a_empty = a_full + RAC;
    uint64_t* acc_full = a_empty + RAC;
    uint64_t* ss_ready = acc_full + 1;
    uint64_t* g_full = ss_ready + 1;
    uint64_t* tmem_ready = g_full + 1;
    uint64_t* h_all = tmem_ready + 1;                           // first RH blocks landed (cp.async path)
    uint64_t* h_tma = h_all + 1;                                // first RH blocks landed (TMA path)
    int64_t* s_ioff = reinterpret_cast<int64_t*>(h_tma + 1);    // item part of the cache offset, or -1
    int* s_pos = reinterpret_cast<int*>(s_ioff + MAX_ITEMS);
    float* s_ss = reinterpret_cast<float*>(s_pos + MAX_ITEMS);    // partial sum(h^2) over this CTA's k
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s_ss + MAX_ITEMS);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    float* ptile = reinterpret_cast<float*>(smem + Lay::OFF_H);  // epilogue [item][P_LD] (after the last MMA)

    const int ks = a.ks;
    const int rank = static_cast<int>(cluster_rank());
    const int tile = blockIdx.x / ks, li = blockIdx.y;
    const DecodeLayer& L = a.l[li];
    const bool is_k = tile < a.tpk;
    const int kv = is_k ? 0 : 1;
    const int tk = is_k ? tile : tile - a.tpk;        // tile within the K (or V) projection
    // A K-only or V-only layer: the other kind's clusters leave before any shared state.
    if (L.writes == (is_k ? TEE_FILL_WRITE_V : TEE_FILL_WRITE_K)) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nbc = a.nb / ks, k0 = rank * nbc * KB;     // this CTA's blocks and first k
    const int nch = (nbc + CHB - 1) / CHB;
    const int pre = min(Lay::RH, nbc);                   // blocks of h in the first request
    const uint8_t* wsrc = L.w + (static_cast<int64_t>(kv * a.tpk + tk) * a.nb + rank * nbc) * BLK_BYTES;
    // one CTA (the first that runs for layer 0) records bad rows / positions
    const bool reporter = li == 0 && rank == 0 && tile == (a.l[0].writes == TEE_FILL_WRITE_V ? a.tpk : 0);

    if (warp == LD_WARP) {
        // Lane 0 sets up what the weight copies need and starts them at once (the
        // weights are constant: they stream in before the previous kernel has
        // finished, with an early launch); the other lanes set up the rest.
        if (lane == 0) {
            for (int s = 0; s < RW; ++s) tc::mbar_init(&w_full[s], 1);   // expect_tx + the copy's bytes
            tc::mbar_init(g_full, 1);
            tc::fence_barrier_init();
            // g_j over the k range first: the copy engine serves copies in order
            tc::mbar_arrive_expect_tx(g_full, static_cast<uint32_t>(nbc * KB * 2));
            bulk_load(smem + Lay::OFF_G, L.gamma + k0, static_cast<uint32_t>(nbc * KB * 2), g_full);
            for (int c = 0; c < RW && c < nch; ++c) {
                const uint32_t bytes = static_cast<uint32_t>(min(CHB, nbc - c * CHB)) * BLK_BYTES;
                tc::mbar_arrive_expect_tx(&w_full[c], bytes);
                bulk_load(smem + Lay::OFF_W + c * CHUNK_BYTES, wsrc + static_cast<int64_t>(c) * CHUNK_BYTES, bytes,
                          &w_full[c]);
            }
        } else {
            for (int s = lane - 1; s < Lay::RH; s += 31) {
                tc::mbar_init(&h_full[s], CP_WARPS);
                tc::mbar_init(&h_empty[s], 1);               // MMA commit
            }
            if (lane <= RW) tc::mbar_init(&w_empty[lane - 1], DEQ_WARPS);
            if (lane <= RAC) {
                tc::mbar_init(&a_full[lane - 1], DEQ_WARPS);   // every dequantising warp, once per chunk
                tc::mbar_init(&a_empty[lane - 1], 1);          // MMA commit
            }
            if (lane == 8) tc::mbar_init(acc_full, 1);
            if (lane == 9) tc::mbar_init(ss_ready, CP_WARPS);
            if (lane == 10) tc::mbar_init(tmem_ready, 1);
            if (lane == 11) tc::mbar_init(h_all, H_WARPS);
            if (lane == 12) tc::mbar_init(h_tma, 1);
            if (lane == 14) *abort = 0;
            tc::fence_barrier_init();
        }
        __syncwarp();
    }
    for (int i = threadIdx.x; i < MAX_ITEMS; i += THREADS) s_ss[i] = 0.f;
    __syncthreads();   // barriers initialised
    // Tensor memory is allocated while h streams in; its users wait for tmem_ready.
    if (warp == MMA_WARP) {
        tc::tmem_alloc(tmem_slot, TMEM_COLS);
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(tmem_ready);
    }
    // ---- the items' h rows of the first `pre` blocks. Contiguous rows (a batch
    // whose tokens all exit, or any compacted buffer): one TMA copy by warp 17.
    // Otherwise every warp that has nothing else to do yet requests 16-byte pieces
    // with cp.async (the copy rate per SM grows with the number of warps issuing)
    // and arrives on h_all once its own have landed.
    wait_prior_grid();
    const int n = min(item_count(a.n_max, a.n_dev), Lay::ITEMS);
    int r0 = 0;
    const bool contig = a.h_tma && rows_contiguous(a, n, lane, r0);
    if (warp == LD_WARP) {
        if (contig && lane == 0) {
            tc::mbar_arrive_expect_tx(h_tma, static_cast<uint32_t>(pre) * Lay::H_SLOT);
            tc::tma_load_3d(smem + Lay::OFF_H, &tm_h, 0, r0, k0 / KB, h_tma);
        }
        __syncwarp();
    } else if (warp != MMA_WARP && !contig) {
        const int hw = warp < DEQ_WARPS ? warp : DEQ_WARPS + (warp - CP_WARP0);
        for (int pc = hw * 32 + lane; pc < pre * n * 8; pc += H_WARPS * 32) {
            const int blk = pc / (n * 8), rem = pc - blk * (n * 8), i = rem >> 3, j = rem & 7;
            const int r = a.rows ? a.rows[i] : i;
            if (r >= 0 && r < a.h_rows)
                cp_async16(smem + Lay::OFF_H + blk * Lay::H_SLOT + i * 128 + ((j ^ (i & 7)) << 4),
                           a.h + static_cast<int64_t>(r) * a.ld_h + k0 + blk * KB + j * 8);
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(h_all);
    }
    uint32_t tmem = 0;
    if (warp <= MMA_WARP) {
        warp_wait(tmem_ready, 0, abort, ws, 60);
        tc::tc_fence_after();
        tmem = *tmem_slot;
    }

    if (warp < DEQ_WARPS) {
        bool ok = warp_wait(g_full, 0, abort, ws, 69);
        // ---- dequantise: thread = tile column 32 q + lane, block j of each chunk
        const int q = warp & 3, j = warp >> 2;
        const int col = 32 * q + lane;
        const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
        for (int c = 0; c < nch && ok; ++c) {
            const int slot = c % RW;
            if (!warp_wait(&w_full[slot], (c / RW) & 1, abort, ws, 61)) {
                ok = false;
                break;
            }
            // the chunk's A slots (tensor memory), once the MMAs of two chunks back are done
            const int ac = c % RAC;
            if (c >= RAC && !warp_wait(&a_empty[ac], ((c / RAC) - 1) & 1, abort, ws, 62)) {
                ok = false;
                break;
            }
            const int kb = c * CHB + j;
            if (kb < nbc) {
                const int sa = ac * CHB + j;
                const uint8_t* blk = smem + Lay::OFF_W + slot * CHUNK_BYTES + j * BLK_BYTES;
                const uint4 c0 = *reinterpret_cast<const uint4*>(blk + col * 16);
                const uint4 c1 = *reinterpret_cast<const uint4*>(blk + CODE_HALF + col * 16);
                const uint32_t sc = *reinterpret_cast<const uint32_t*>(blk + SC_OFF + col * 4);
                const uint32_t s_w = __byte_perm(sc, 0, 0x1010), c_w = __byte_perm(sc, 0, 0x3232);
                const __nv_bfloat162 s2 = *reinterpret_cast<const __nv_bfloat162*>(&s_w);
                const __nv_bfloat162 c2 = *reinterpret_cast<const __nv_bfloat162*>(&c_w);
                // g_j of the block's 64 k as bf16 pairs (the same for every lane)
                const uint4* gp = reinterpret_cast<const uint4*>(smem + Lay::OFF_G + kb * KB * 2);
                uint32_t o[32];
                deq_word(c0.x, s2, c2, gp[0], o + 0);
                deq_word(c0.y, s2, c2, gp[1], o + 4);
                deq_word(c0.z, s2, c2, gp[2], o + 8);
                deq_word(c0.w, s2, c2, gp[3], o + 12);
                deq_word(c1.x, s2, c2, gp[4], o + 16);
                deq_word(c1.y, s2, c2, gp[5], o + 20);
                deq_word(c1.z, s2, c2, gp[6], o + 24);
                deq_word(c1.w, s2, c2, gp[7], o + 28);
                tmem_st32(tmem + lane_base + ACC_COLS + 32 * sa, o);
                tmem_st_wait();
            }
            // One hand-over per chunk: the MMA issuer's tcgen05 fence after its wait
            // drains the tensor pipe, so it is paid once for four blocks.
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                tc::mbar_arrive(&a_full[ac]);
                tc::mbar_arrive(&w_empty[slot]);   // this warp is done with the chunk
            }
        }
    } else if (warp == MMA_WARP) {
        // ---- MMA issuer: N = the items rounded up to 16
        if (lane == 0) {
            wait_prior_grid();
            const int nn = max(16, (min(item_count(a.n_max, a.n_dev), Lay::ITEMS) + 15) & ~15);
            const uint32_t idesc = tc::idesc_bf16(T_COLS, nn);
            bool ok = tc::mbar_wait(contig ? h_tma : h_all, 0, abort, ws, 64);
            for (int c = 0; c < nch && ok; ++c) {
                const int ac = c % RAC;
                if (!tc::mbar_wait(&a_full[ac], (c / RAC) & 1, abort, ws, 63)) break;
                for (int kb = c * CHB; kb < min(nbc, (c + 1) * CHB) && ok; ++kb) {
                    const int sh = kb % Lay::RH;
                    if (kb >= Lay::RH && !tc::mbar_wait(&h_full[sh], ((kb / Lay::RH) - 1) & 1, abort, ws, 64)) {
                        ok = false;
                        break;
                    }
                }
                if (!ok) break;
                tc::tc_fence_after();   // once per chunk (it waits for the tensor pipe)
                for (int kb = c * CHB; kb < min(nbc, (c + 1) * CHB); ++kb) {
                    const int sa = ac * CHB + (kb - c * CHB), sh = kb % Lay::RH;
                    const uint64_t bd = tc::smem_desc_sw128(tc::smem_u32(smem + Lay::OFF_H + sh * Lay::H_SLOT));
#pragma unroll
                    for (int kk = 0; kk < KB / 16; ++kk)
                        umma_ts(tmem, tmem + ACC_COLS + 32 * sa + 8 * kk, bd + 2 * kk, idesc, kb | kk);
                    tc::umma_commit(&h_empty[sh]);
                }
                tc::umma_commit(&a_empty[ac]);
            }
            tc::umma_commit(acc_full);   // also when stopped early: every issued MMA finishes first
        }
        __syncwarp();
    } else if (warp == LD_WARP) {
        // ---- weight chunks beyond the first RW
        if (lane == 0) {
            for (int c = RW; c < nch; ++c) {
                const int slot = c % RW;
                if (!tc::mbar_wait(&w_empty[slot], ((c / RW) - 1) & 1, abort, ws, 65)) break;
                const uint32_t bytes = static_cast<uint32_t>(min(CHB, nbc - c * CHB)) * BLK_BYTES;
                tc::mbar_arrive_expect_tx(&w_full[slot], bytes);
                bulk_load(smem + Lay::OFF_W + slot * CHUNK_BYTES, wsrc + static_cast<int64_t>(c) * CHUNK_BYTES, bytes,
                          &w_full[slot]);
            }
        }
        __syncwarp();
    } else {
        // ---- cache slots, sums of h^2 and, past the first RH blocks (a long k
        // range), the B ring. Thread ct owns 16-byte piece j = ct % 8 of items
        // ct / 8 + 16 m.
        const int ct = threadIdx.x - CP_WARP0 * 32;
        const int j = ct & 7, ib = ct >> 3;
        int r_ct = -1;
        if (ct < n) {
            const int r = a.rows ? a.rows[ct] : ct;
            if (r >= 0 && r < a.h_rows) r_ct = r;
            else if (reporter) record_fault(ws, TEE_DEVERR_ROW, r);
        }
        // Item ct's position and cache slot; the RoPE row it needs into L2.
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
                    if (is_k) {   // plain line prefetches (bulk ones would queue behind the weight copies)
                        const char* rp = reinterpret_cast<const char*>(a.rope + static_cast<int64_t>(p) * a.half);
                        for (int o = 0; o < a.half * 8; o += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(rp + o));
                    }
                }
            }
            s_ioff[ct] = ioff;
            s_pos[ct] = p;
        }
        // Sums of h^2 over this CTA's k range, read from the B operands once they
        // have landed (read-only: the MMA reads the same blocks meanwhile).
        float ss[Lay::IPC];
#pragma unroll
        for (int m = 0; m < Lay::IPC; ++m) ss[m] = 0.f;
        bool valid[Lay::IPC];
#pragma unroll
        for (int m = 0; m < Lay::IPC; ++m) {
            const int i = ib + 16 * m;
            const int r = i < n ? (a.rows ? a.rows[i] : i) : -1;
            valid[m] = r >= 0 && r < a.h_rows;
        }
        bool ok = warp_wait(contig ? h_tma : h_all, 0, abort, ws, 70);
        if (ok) {
            for (int b = 0; b < pre; ++b) {
                const uint8_t* slot = smem + Lay::OFF_H + b * Lay::H_SLOT;
#pragma unroll
                for (int m = 0; m < Lay::IPC; ++m) {
                    const int i = ib + 16 * m;
                    if (valid[m]) ss[m] = sumsq8(*reinterpret_cast<const uint4*>(slot + i * 128 + ((j ^ (i & 7)) << 4)), ss[m]);
                }
            }
        }
        // Blocks past the first RH (a long k range) through the ring.
        for (int kb = pre; kb < nbc && ok; ++kb) {
            const int s = kb % Lay::RH;
            if (!warp_wait(&h_empty[s], ((kb / Lay::RH) - 1) & 1, abort, ws, 66)) {   // the MMA read kb - RH
                ok = false;
                break;
            }
            uint8_t* slot = smem + Lay::OFF_H + s * Lay::H_SLOT;
#pragma unroll
            for (int m = 0; m < Lay::IPC; ++m) {
                const int i = ib + 16 * m;
                if (valid[m])
                    cp_async16(slot + i * 128 + ((j ^ (i & 7)) << 4),
                               a.h + static_cast<int64_t>(a.rows ? a.rows[i] : i) * a.ld_h + k0 + kb * KB + j * 8);
            }
            asm volatile("cp.async.wait_all;" ::: "memory");
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&h_full[s]);
#pragma unroll
            for (int m = 0; m < Lay::IPC; ++m) {
                const int i = ib + 16 * m;
                if (valid[m]) ss[m] = sumsq8(*reinterpret_cast<const uint4*>(slot + i * 128 + ((j ^ (i & 7)) << 4)), ss[m]);
            }
        }
#pragma unroll
        for (int m = 0; m < Lay::IPC; ++m) {   // the eight threads of an item are consecutive lanes
            float t = ss[m];
            t += __shfl_xor_sync(0xffffffffu, t, 1);
            t += __shfl_xor_sync(0xffffffffu, t, 2);
            t += __shfl_xor_sync(0xffffffffu, t, 4);
            if (j == 0) s_ss[ib + 16 * m] = t;
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(ss_ready);   // release: s_ss, s_ioff, s_pos are ready
    }

    // ---- accumulator -> [item][column] tile in shared memory (the B ring's space)
    bool acc_ok = true;
    if (warp < DEQ_WARPS) {
        acc_ok = warp_wait(acc_full, 0, abort, ws, 67);
        acc_ok = warp_wait(ss_ready, 0, abort, ws, 68) && acc_ok;   // s_ss, s_ioff, s_pos
        tc::tc_fence_after();
        const int q = warp & 3, j = warp >> 2;
        const uint32_t tb = tmem + (static_cast<uint32_t>(32 * q) << 16) + j * Lay::IPW;
        const int col = 32 * q + lane;
        if (acc_ok) {
            if constexpr (Lay::IPW == 16) {
                float v[16];
                tc::tmem_ld16(tb, v);
#pragma unroll
                for (int e = 0; e < 16; ++e) ptile[(j * 16 + e) * P_LD + col] = v[e];
            } else {
                float v[32];
                tc::tmem_ld32(tb, v);
#pragma unroll
                for (int e = 0; e < 32; ++e) ptile[(j * 32 + e) * P_LD + col] = v[e];
            }
        }
    }
    tc::tc_fence_before();
    cluster_sync();   // every CTA's tile and partial sums of h^2 are complete
    tc::tc_fence_after();

    // ---- finish the items of this rank: thread = (item, 8 rotation pairs), eight
    // threads per item (a tile's 128 columns are 64 pairs of whole heads).
    if (warp < DEQ_WARPS && acc_ok && !*abort) {
        const int own = Lay::ITEMS / ks;          // items finished per CTA
        const int spp = a.hd / 16;                // 8-pair segments per head
        const bf16* bias = L.bias[kv];
        const bool knorm = is_k && L.k_norm;
        const unsigned gmask = (spp == 4 ? 0xFu : 0xFFu) << (lane & (spp == 4 ? 28 : 24));
        for (int task = threadIdx.x; task < own * 8; task += DEQ_THREADS) {
            const int i = rank * own + (task >> 3), seg = task & 7;
            // the eight threads of an item agree on skipping it (shuffles below)
            if (i >= n || s_ioff[i] < 0) continue;
            const int64_t ioff = s_ioff[i];
            const int hh = seg / spp, p0 = 8 * (seg % spp);
            const int c_lo = hh * a.hd + p0, c_hi = c_lo + a.half;   // tile columns
            float4 c2[4];   // {cos, sin} of the 8 pairs (K only), loaded first: the longest latency
            if (is_k) {
                const float4* cs = reinterpret_cast<const float4*>(a.rope + static_cast<int64_t>(s_pos[i]) * a.half + p0);
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) c2[e2] = __ldg(cs + e2);
            }
            float ssum = s_ss[i];
            float lo[8], hi[8];
            {
                const float4* pl = reinterpret_cast<const float4*>(ptile + i * P_LD + c_lo);
                const float4* ph = reinterpret_cast<const float4*>(ptile + i * P_LD + c_hi);
                float4 v[4] = {pl[0], pl[1], ph[0], ph[1]};
                for (int r = 0; r < ks; ++r) {   // the peers' partials, all loads before use
                    if (r == rank) continue;
                    const uint32_t bl = peer_addr(ptile + i * P_LD + c_lo, r);
                    const uint32_t bh = peer_addr(ptile + i * P_LD + c_hi, r);
                    const float4 u0 = ld_peer_f4(bl), u1 = ld_peer_f4(bl + 16);
                    const float4 u2 = ld_peer_f4(bh), u3 = ld_peer_f4(bh + 16);
                    ssum += ld_peer_f32(peer_addr(s_ss + i, r));
                    v[0].x += u0.x; v[0].y += u0.y; v[0].z += u0.z; v[0].w += u0.w;
                    v[1].x += u1.x; v[1].y += u1.y; v[1].z += u1.z; v[1].w += u1.w;
                    v[2].x += u2.x; v[2].y += u2.y; v[2].z += u2.z; v[2].w += u2.w;
                    v[3].x += u3.x; v[3].y += u3.y; v[3].z += u3.z; v[3].w += u3.w;
                }
                lo[0] = v[0].x; lo[1] = v[0].y; lo[2] = v[0].z; lo[3] = v[0].w;
                lo[4] = v[1].x; lo[5] = v[1].y; lo[6] = v[1].z; lo[7] = v[1].w;
                hi[0] = v[2].x; hi[1] = v[2].y; hi[2] = v[2].z; hi[3] = v[2].w;
                hi[4] = v[3].x; hi[5] = v[3].y; hi[6] = v[3].z; hi[7] = v[3].w;
            }
            const float rs = 1.0f / sqrtf(ssum * a.inv_d + a.eps);
            const int gcol = tk * T_COLS + c_lo;    // column within the K (or V) projection
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                lo[e] *= rs;
                hi[e] *= rs;
            }
            if (bias) {
                float b[8];
                load8_bf16(bias + gcol, b);
#pragma unroll
                for (int e = 0; e < 8; ++e) lo[e] += b[e];
                load8_bf16(bias + gcol + a.half, b);
#pragma unroll
                for (int e = 0; e < 8; ++e) hi[e] += b[e];
            }
            if (knorm) {
                // the head's RMS over its hd values: the spp threads of the head
                float hss = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) hss = fmaf(lo[e], lo[e], fmaf(hi[e], hi[e], hss));
                hss += __shfl_xor_sync(gmask, hss, 1);
                hss += __shfl_xor_sync(gmask, hss, 2);
                if (spp == 8) hss += __shfl_xor_sync(gmask, hss, 4);
                const float hs = 1.0f / sqrtf(hss / static_cast<float>(a.hd) + a.eps);
                float g[8];
                load8_bf16(L.k_norm + p0, g);
#pragma unroll
                for (int e = 0; e < 8; ++e) lo[e] *= hs * g[e];
                load8_bf16(L.k_norm + a.half + p0, g);
#pragma unroll
                for (int e = 0; e < 8; ++e) hi[e] *= hs * g[e];
            }
            if (is_k) {
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) {   // pairs p0 + 2 e2, + 1
                    const float x1 = lo[2 * e2], x2 = hi[2 * e2];
                    const float y1 = lo[2 * e2 + 1], y2 = hi[2 * e2 + 1];
                    lo[2 * e2] = x1 * c2[e2].x - x2 * c2[e2].y;
                    hi[2 * e2] = x2 * c2[e2].x + x1 * c2[e2].y;
                    lo[2 * e2 + 1] = y1 * c2[e2].z - y2 * c2[e2].w;
                    hi[2 * e2 + 1] = y2 * c2[e2].z + y1 * c2[e2].w;
                }
            }
            const int head = gcol / a.hd;
            bf16* dst = (is_k ? a.kc : a.vc) + ioff + static_cast<int64_t>(head) * a.cl.s_head + p0;
            *reinterpret_cast<uint4*>(dst) = make_uint4(pack_bf16x2(lo[0], lo[1]), pack_bf16x2(lo[2], lo[3]),
                                                        pack_bf16x2(lo[4], lo[5]), pack_bf16x2(lo[6], lo[7]));
            *reinterpret_cast<uint4*>(dst + a.half) = make_uint4(pack_bf16x2(hi[0], hi[1]), pack_bf16x2(hi[2], hi[3]),
                                                                 pack_bf16x2(hi[4], hi[5]), pack_bf16x2(hi[6], hi[7]));
        }
    }
    // No CTA leaves while a peer may still read its tile: arrive now (this CTA's
    // reads of its peers are done), wait just before leaving.
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("cp.async.wait_all;" ::: "memory");
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == MMA_WARP) tc::tmem_dealloc(tmem, TMEM_COLS);
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- prepare
// One thread per (tile, block, column) of one projection: the column's 64 codes
// of the block in the kernel's nibble order, and its bf16 s and (8 - z) s
// (computed in fp32), into the block's record.
__global__ void decode_repack_kernel(const uint8_t* __restrict__ codes, const __half* __restrict__ scale,
                                     const __half* __restrict__ zero, int kvw, int nb, uint8_t* __restrict__ out) {
    const int64_t total = static_cast<int64_t>(kvw / T_COLS) * nb * T_COLS;
    for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int c = static_cast<int>(idx % T_COLS);
        const int b = static_cast<int>((idx / T_COLS) % nb);
        const int tk = static_cast<int>(idx / (static_cast<int64_t>(T_COLS) * nb));
        const int col = tk * T_COLS + c;
        uint8_t* rec = out + (static_cast<int64_t>(tk) * nb + b) * BLK_BYTES;
        uint32_t wd[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {   // word i: k 8 i .. 8 i + 7 of the block
            uint32_t w = 0;
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const uint8_t byte = codes[static_cast<int64_t>(b * (KB / 2) + 4 * i + p) * kvw + col];
                w |= static_cast<uint32_t>(byte & 0xF) << (4 * p);          // k = 8 i + 2 p
                w |= static_cast<uint32_t>(byte >> 4) << (16 + 4 * p);      // k = 8 i + 2 p + 1
            }
            wd[i] = w;
        }
        *reinterpret_cast<uint4*>(rec + c * 16) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
        *reinterpret_cast<uint4*>(rec + CODE_HALF + c * 16) = make_uint4(wd[4], wd[5], wd[6], wd[7]);
        const float s = __half2float(scale[static_cast<int64_t>(b) * kvw + col]);
        const float z = __half2float(zero[static_cast<int64_t>(b) * kvw + col]);
        *reinterpret_cast<uint32_t*>(rec + SC_OFF + c * 4) = pack_bf16x2(s, (8.0f - z) * s);
    }
}

bool desc_ok(const tee_fill_desc& D) {
    const int kvw = D.n_kv_heads * D.head_dim;
    return D.dtype == TEE_BF16 && D.wfmt == TEE_W_INT4 && D.group == KB && D.d % KB == 0 &&
           (D.head_dim == 64 || D.head_dim == 128) && kvw % T_COLS == 0;
}

size_t layer_rec_bytes(const tee_fill_desc& D) {
    const size_t kvw = static_cast<size_t>(D.n_kv_heads) * D.head_dim;
    return 2 * (kvw / T_COLS) * (D.d / KB) * BLK_BYTES;
}

bool decode_eligible(const FillCall& fc) {
    const tee_fill_desc& D = *fc.desc;
    if (!desc_ok(D)) return false;
    if (fc.n_max > MAX_ITEMS || fc.n_layers > MAX_DECODE_LAYERS) return false;
    if ((fc.ld_h * 2) % 16 || !aligned16(fc.h) || !aligned16(fc.k_cache) || !aligned16(fc.v_cache)) return false;
    const tee_cache_layout& cl = *fc.cache;
    if (cl.s_layer % 8 || cl.s_seq % 8 || cl.s_head % 8 || cl.s_pos % 8) return false;
    for (int l = 0; l < fc.n_layers; ++l) {
        const tee_fill_layer& L = fc.layers[l];
        if (L.w_map || !aligned16(L.gamma)) return false;
    }
    return true;
}

template <bool NARROW>
tee_status launch(const CUtensorMap& tm, DecodeArgs a, dim3 grid, int ks, bool early, void* ws, cudaStream_t stream) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(THREADS);
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
    // h as rows x 64-k blocks, box = the items' rows x the blocks of the first request
    const int pre = a.nb / ks < DLayout<NARROW>::RH ? a.nb / ks : DLayout<NARROW>::RH;
    CUtensorMap map = tm;
    a.h_tma = a.h_rows > 0 && make_tmap_bf16_kblocks(&map, a.h, static_cast<uint64_t>(a.h_rows),
                                                     static_cast<uint64_t>(a.ld_h) * 2, static_cast<uint64_t>(a.nb),
                                                     DLayout<NARROW>::ITEMS, static_cast<uint32_t>(pre)) == TEE_OK;
    const tee_status st = cuda_status(cudaLaunchKernelEx(&cfg, fill_decode_kernel<NARROW>, map, a, ws));
    return st != TEE_OK ? st : launch_status();   // counts the launch
}

// Clusters of ks CTAs that can be resident at once (one CTA per SM either way).
int max_clusters(int ks) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(ks * 64, 1);
    cfg.blockDim = dim3(THREADS);
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

// K split: the largest of 4, 2, 1 that divides the 64-k blocks evenly and keeps
// the grid within the SMs and the clusters that can be resident at once.
int choose_ks(int nb, int tiles, int mc4, int mc2) {
    const int sms = sm_count();
    if (nb % 4 == 0 && ((tiles * 4 <= sms && tiles <= mc4) || nb / 2 > MAX_NBC)) return 4;
    if (nb % 2 == 0 && ((tiles * 2 <= sms && tiles <= mc2) || nb > MAX_NBC)) return 2;
    return 1;
}

}  // namespace

size_t fill_decode_prep_bytes(const tee_fill_desc& D, int n_layers) {
    if (!desc_ok(D)) return 0;
    return static_cast<size_t>(n_layers) * layer_rec_bytes(D);
}

tee_status fill_decode_prepare(const tee_fill_desc& D, int n_layers, const tee_fill_layer* layers, char* area,
                               cudaStream_t s) {
    if (!desc_ok(D)) return TEE_OK;
    const int kvw = D.n_kv_heads * D.head_dim, nb = D.d / KB;
    const size_t half = layer_rec_bytes(D) / 2;
    for (int l = 0; l < n_layers; ++l) {
        const tee_fill_layer& L = layers[l];
        if (!L.wk || !L.wv || !L.k_scale || !L.k_zero || !L.v_scale || !L.v_zero) return TEE_ERR_INVALID_ARG;
        uint8_t* base = reinterpret_cast<uint8_t*>(area + l * layer_rec_bytes(D));
        const int64_t total = static_cast<int64_t>(kvw / T_COLS) * nb * T_COLS;
        const int blocks = static_cast<int>((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
        decode_repack_kernel<<<blocks, 256, 0, s>>>(static_cast<const uint8_t*>(L.wk),
                                                    static_cast<const __half*>(L.k_scale),
                                                    static_cast<const __half*>(L.k_zero), kvw, nb, base);
        tee_status st = launch_status();
        if (st != TEE_OK) return st;
        decode_repack_kernel<<<blocks, 256, 0, s>>>(static_cast<const uint8_t*>(L.wv),
                                                    static_cast<const __half*>(L.v_scale),
                                                    static_cast<const __half*>(L.v_zero), kvw, nb, base + half);
        st = launch_status();
        if (st != TEE_OK) return st;
    }
    return TEE_OK;
}

size_t fill_decode_ws_bytes(const tee_fill_desc&, int, int) { return TEE_WS_HEADER_BYTES; }

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
    a.tpk = a.kvw / T_COLS;
    a.nb = D.d / KB;
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
        a.l[l] = DecodeLayer{reinterpret_cast<const uint8_t*>(pv.dec) + l * layer_rec_bytes(D),
                             static_cast<const bf16*>(L.gamma),
                             {static_cast<const bf16*>(L.k_bias), static_cast<const bf16*>(L.v_bias)},
                             static_cast<const bf16*>(L.k_norm), L.cache_layer, L.writes};
    }
    const int tiles = 2 * a.tpk * fc.n_layers;   // (tile, layer) pairs
    a.ks = choose_ks(a.nb, tiles, mc4, mc2);
    if (a.nb / a.ks > MAX_NBC) return TEE_ERR_UNSUPPORTED;
    const dim3 grid(2 * a.tpk * a.ks, fc.n_layers);
    // An early launch parks the grid's CTAs on their SMs until the previous kernel
    // completes: only when the grid leaves SMs free for that kernel to finish on.
    const bool early = (D.flags & TEE_FILL_EARLY_WEIGHTS) && static_cast<int>(grid.x * grid.y) + 4 <= sm_count();
    CUtensorMap tm{};
    return fc.n_max <= DLayout<true>::ITEMS ? launch<true>(tm, a, grid, a.ks, early, fc.ws, fc.stream)
                                            : launch<false>(tm, a, grid, a.ks, early, fc.ws, fc.stream);
}

}  // namespace tee
