// TIDE router gate on tcgen05 for large batches (formula 3; module 4
// "Fused LayerNorm + Route"): the whole gate in one launch.
//
//   dots[t][c] = sum_i W_down[c][i] h[t][i],  sumsq[t] = sum_i h[t][i]^2,
//   p[t] = sigmoid(b_up + sum_c w_up[c] SiLU(dots[t][c] / rms(h[t]) + b_down[c])),
//   mask[t] = p[t] > theta.
//
// M = 128 tokens x N = 128 router channels per tile; K = d split over KS CTAs so
// that the batch spreads over the SMs. The KS CTAs of a token tile form a
// cluster. In each CTA, warp 4 streams 128x64 tiles of h and W_down (already
// K-major: TMA reads the caller's array) into a 6-stage ring (128-byte swizzle),
// one thread of warp 5 issues tcgen05.mma into a 128-column TMEM accumulator,
// and warps 0-3 add up sum(h^2) of their token row from each staged h tile (the
// fused RMSNorm; a ring slot is freed by the MMA commit plus the four warps).
// Then warps 0-3 store the partial dots (staged through shared memory, so that
// each row goes out as one coalesced 512-byte store) and the partial sums of h^2
// into the workspace; one cluster barrier (release / acquire at cluster scope);
// each CTA then finishes 128 / KS of the tile's tokens from L2: sums of the KS
// partials, 1/rms, b_down, SiLU, w_up, sigmoid, threshold. The all-tokens flag
// is reduced by the last CTA to finish.
#include "tc.cuh"

namespace tee {

namespace {

using bf16 = __nv_bfloat16;

constexpr int RBM = 128, RBN = 128, RBK = 64;
// A ring stage holds RKZ consecutive 64-k blocks of h and of W_down, each operand
// brought by one TMA copy (a copy costs about the same whatever its size).
constexpr int RKZ = 2, RSTAGES = 3;
constexpr int RTHREADS = 6 * 32;
constexpr int RMAX_SPLIT = 4;   // K split and cluster size at most (keeps the finishing loads in registers)
constexpr uint32_t RA_BYTES = RBM * RBK * 2, RB_BYTES = RBN * RBK * 2;   // one 64-k block
constexpr uint32_t RA_STAGE = RKZ * RA_BYTES, RSTAGE = RKZ * (RA_BYTES + RB_BYTES);   // [A blocks | B blocks]
constexpr int RSTAGE_LD = 132;  // floats per staged row (conflict-free 16-byte stores)
constexpr uint32_t RSTAGING = 4 * 32 * RSTAGE_LD * 4;   // epilogue staging: reuses the ring once the MMAs are done
static_assert(RSTAGING <= RSTAGES * RSTAGE, "staging must fit in the ring");
constexpr size_t RSMEM = 1024 + size_t(RSTAGES) * RSTAGE + 256;
// Smallest batch that goes to the tensor cores.
constexpr int RTC_MIN_TOKENS = 256;

struct RouterArgs {
    int n, d, nks;         // nks: k stages (RKZ blocks of 64 columns) over d
    float eps, thr;
    int rule;
    bool need_flag;
    float* part;           // workspace: [tile][split][128 tokens][128 channels] partial dots
    float* part_ss;        // workspace: [tile][split][128] partial sums of h^2
    const float* b_down;   // [128] or null
    const bf16* w_up;      // [128]
    const float* b_up;     // [1] or null
    float* score;
    uint8_t* mask;
    int32_t* flag;
    float* block_mins;     // workspace: one float per CTA
    uint32_t* counter;     // workspace: CTAs finished
};

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// L2-only loads of what peer CTAs stored before the cluster barrier.
__device__ __forceinline__ float4 ld_l2_f4(const float* p) {
    float4 v;
    asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ float ld_l2_f32(const float* p) {
    float v;
    asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

// All-tokens flag: each CTA publishes the minimum score its warps saw (cmin: this
// warp's); the last CTA to arrive reduces the minima, writes the flag and, under
// the batch rule, the mask of every token. Called by every thread of the CTA.
template <int NT>
__device__ __noinline__ void flag_tail(float cmin, const RouterArgs& a) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __shared__ float s_min[NT / 32];
    __shared__ int s_last;
    if (lane == 0) s_min[warp] = cmin;
    __syncthreads();
    const int nblocks = gridDim.x * gridDim.y, bid = blockIdx.y * gridDim.x + blockIdx.x;
    if (threadIdx.x == 0) {
        float m = INFINITY;
        for (int w = 0; w < NT / 32; ++w) m = fminf(m, s_min[w]);
        a.block_mins[bid] = m;
        __threadfence();
        s_last = atomicAdd(a.counter, 1u) == static_cast<unsigned>(nblocks - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    float m = INFINITY;
    for (int i = threadIdx.x; i < nblocks; i += NT) m = fminf(m, *reinterpret_cast<volatile float*>(a.block_mins + i));
    m = warp_min(m);
    if (lane == 0) s_min[warp] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float mm = INFINITY;
        for (int w = 0; w < NT / 32; ++w) mm = fminf(mm, s_min[w]);
        s_min[0] = mm;
    }
    __syncthreads();
    const uint8_t f = (a.n > 0 && s_min[0] > a.thr) ? 1 : 0;
    if (threadIdx.x == 0) {
        if (a.flag) *a.flag = f;
        *a.counter = 0u;
    }
    if (a.rule == TEE_RULE_BATCH_ALL)
        for (int t = threadIdx.x; t < a.n; t += NT) a.mask[t] = f;
}

__global__ void __launch_bounds__(RTHREADS, 1)
router_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ RouterArgs a, void* ws) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* staging = reinterpret_cast<float*>(smem);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + RSTAGES * RSTAGE);
    uint64_t* empty = full + RSTAGES;
    uint64_t* acc_full = empty + RSTAGES;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x, ks = gridDim.y, split = static_cast<int>(cluster_rank());
    const int m0 = tile * RBM;
    // balanced K split: every split gets at least one stage (splits <= nks / 2)
    const int kb0 = split * a.nks / ks;
    const int kb1 = (split + 1) * a.nks / ks;
    allow_dependents();

    if (threadIdx.x == 0) {
        for (int s = 0; s < RSTAGES; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1 + 4);   // MMA commit + the four sum(h^2) warps
        }
        tc::mbar_init(acc_full, 1);
        *abort = 0;
        tc::fence_barrier_init();
    }
    if (warp == 5) tc::tmem_alloc(tmem_slot, RBN);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    float* part = a.part + static_cast<int64_t>(tile * ks + split) * RBM * RBN;
    float* part_ss = a.part_ss + static_cast<int64_t>(tile * ks + split) * RBM;
    bool ok = true;
    if (warp == 4) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_phase = 0;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!tc::mbar_wait(&empty[stage], phase ^ 1, abort, ws, 31)) break;
                uint8_t* sa = smem + stage * RSTAGE;
                tc::mbar_arrive_expect_tx(&full[stage], RSTAGE);
                tc::tma_load_3d(sa, &tmA, 0, m0, kb * RKZ, &full[stage]);
                tc::tma_load_3d(sa + RA_STAGE, &tmB, 0, 0, kb * RKZ, &full[stage]);
                issued |= 1u << stage;
                issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                if (++stage == RSTAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (*abort) {   // let the copies already issued land before the block moves on
                for (int s = 0; s < RSTAGES; ++s) {
                    if (!(issued >> s & 1)) continue;
                    const uint64_t t0 = tc::globaltimer();
                    while (!tc::mbar_try_wait(&full[s], issued_phase >> s & 1) &&
                           tc::globaltimer() - t0 < tc::WAIT_LIMIT_NS) {
                    }
                }
            }
        }
    } else if (warp == 5) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            constexpr uint32_t idesc = tc::idesc_bf16(RBM, RBN);
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!tc::mbar_wait(&full[stage], phase, abort, ws, 32)) break;
                tc::tc_fence_after();
                const uint32_t sa = tc::smem_u32(smem + stage * RSTAGE);
#pragma unroll
                for (int z = 0; z < RKZ; ++z) {
                    const uint64_t ad = tc::smem_desc_sw128(sa + z * RA_BYTES);
                    const uint64_t bd = tc::smem_desc_sw128(sa + RA_STAGE + z * RB_BYTES);
#pragma unroll
                    for (int k = 0; k < RBK / 16; ++k)
                        tc::umma_bf16(tmem, ad + 2 * k, bd + 2 * k, idesc, (kb - kb0) | z | k);
                }
                tc::umma_commit(&empty[stage]);
                if (++stage == RSTAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            tc::umma_commit(acc_full);  // also when stopped early: every issued MMA finishes first
            // ... and this thread sees it before the block frees TMEM, even after an
            // abort (the wait ignores the flag and ends by its time limit)
            const uint64_t t0 = tc::globaltimer();
            while (!tc::mbar_try_wait(acc_full, 0) && tc::globaltimer() - t0 < tc::WAIT_LIMIT_NS) {
            }
        }
    } else {
        // warps 0-3: sum(h^2) of token row (warp*32 + lane) from each staged h tile
        const int r = warp * 32 + lane;
        float ss = 0.f;
        int stage = 0;
        uint32_t phase = 0;
        for (int kb = kb0; kb < kb1; ++kb) {
            if (!__all_sync(0xffffffffu, tc::mbar_wait(&full[stage], phase, abort, ws, 33))) {
                ok = false;
                break;
            }
#pragma unroll
            for (int jj = 0; jj < 8 * RKZ; ++jj) {
                // block jj / 8 of the stage; rotate the chunk order by row: lanes of a
                // warp hit 8 different bank groups
                const int j = jj & 7;
                const uint8_t* row = smem + stage * RSTAGE + (jj >> 3) * RA_BYTES + r * 128;
                const uint4 v = *reinterpret_cast<const uint4*>(row + (((j + r) & 7) << 4));
                float x[8];
                unpack_bf16x2(v.x, x[0], x[1]);
                unpack_bf16x2(v.y, x[2], x[3]);
                unpack_bf16x2(v.z, x[4], x[5]);
                unpack_bf16x2(v.w, x[6], x[7]);
#pragma unroll
                for (int q = 0; q < 8; ++q) ss = fmaf(x[q], x[q], ss);
            }
            // Order these generic-proxy reads before the async-proxy (TMA) refill of the slot.
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&empty[stage]);
            if (++stage == RSTAGES) {
                stage = 0;
                phase ^= 1;
            }
        }
        if (ok) ok = tc::mbar_wait(acc_full, 0, abort, ws, 34);
        ok = __all_sync(0xffffffffu, ok);   // tcgen05.ld below is warp-collective
        tc::tc_fence_after();
        // The staging area overlays the ring: every MMA has read its operands
        // (acc_full), and this barrier waits until the four warps are done with
        // their last tiles. Not .aligned: lanes may leave the loop on a timeout apart.
        asm volatile("barrier.sync 1, 128;" ::: "memory");
        if (ok) {
            // Stage this warp's 32 rows in shared memory (row stride 132 floats keeps
            // the 16-byte stores conflict-free), then store each row with one 512-byte
            // coalesced warp store.
            float* stage_rows = staging + warp * (32 * RSTAGE_LD);
            const uint32_t tb = tmem + (static_cast<uint32_t>(warp * 32) << 16);
#pragma unroll 1
            for (int c = 0; c < RBN; c += 32) {
                float v[32];
                tc::tmem_ld32(tb + c, v);
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    *reinterpret_cast<float4*>(stage_rows + lane * RSTAGE_LD + c + 4 * q) =
                        make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            }
            __syncwarp();
            for (int rr = 0; rr < 32; ++rr)
                *reinterpret_cast<float4*>(part + (warp * 32 + rr) * RBN + lane * 4) =
                    *reinterpret_cast<const float4*>(stage_rows + rr * RSTAGE_LD + lane * 4);
            part_ss[r] = ss;
        }
    }
    // The finishing constants load while the cluster meets.
    const int tq = lane >> 3, cl = lane & 7, c0 = 16 * cl;
    float wu[16], bd[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
        wu[e] = __bfloat162float(a.w_up[c0 + e]);
        bd[e] = a.b_down ? a.b_down[c0 + e] : 0.f;
    }
    const float bu = a.b_up ? a.b_up[0] : 0.f;
    tc::tc_fence_before();
    cluster_sync();   // the tile's partials are visible to every CTA of the cluster
    tc::tc_fence_after();

    // ---- finish tokens m0 + split * T .. + T of the tile (T = 128 / KS). A warp takes
    // four tokens at a time, eight lanes per token, 16 channels per lane.
    const int T = RBM / ks;
    float cmin = INFINITY;
    if (!*abort) {
        const float* tile_part = a.part + static_cast<int64_t>(tile * ks) * RBM * RBN;
        const float* tile_ss = a.part_ss + static_cast<int64_t>(tile * ks) * RBM;
        // Loads of one group (4 tokens of this warp); the next group's loads are in
        // flight while this one is computed.
        float4 pv[2][RMAX_SPLIT][4];
        float sv[2][RMAX_SPLIT];
        auto load_group = [&](int i0, int buf) {
            const int i = i0 + tq, rl = split * T + i, t = m0 + rl;
            if (i >= T || t >= a.n) return;
#pragma unroll
            for (int s2 = 0; s2 < RMAX_SPLIT; ++s2)
                if (s2 < ks) {
                    const float* row = tile_part + (static_cast<int64_t>(s2) * RBM + rl) * RBN + c0;
#pragma unroll
                    for (int e = 0; e < 4; ++e) pv[buf][s2][e] = ld_l2_f4(row + 4 * e);
                    sv[buf][s2] = ld_l2_f32(tile_ss + s2 * RBM + rl);
                }
        };
        constexpr int GSTEP = 4 * (RTHREADS / 32);
        if (4 * warp < T) load_group(4 * warp, 0);
        int buf = 0;
        for (int i0 = 4 * warp; i0 < T; i0 += GSTEP, buf ^= 1) {
            if (i0 + GSTEP < T) load_group(i0 + GSTEP, buf ^ 1);
            const int i = i0 + tq, rl = split * T + i, t = m0 + rl;
            const bool live = i < T && t < a.n;
            float u[16], ss = 0.f;
#pragma unroll
            for (int e = 0; e < 16; ++e) u[e] = 0.f;
#pragma unroll
            for (int s2 = 0; s2 < RMAX_SPLIT; ++s2)
                if (s2 < ks && live) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float4 v = buf ? pv[1][s2][e] : pv[0][s2][e];
                        u[4 * e] += v.x;
                        u[4 * e + 1] += v.y;
                        u[4 * e + 2] += v.z;
                        u[4 * e + 3] += v.w;
                    }
                    ss += buf ? sv[1][s2] : sv[0][s2];
                }
            const float rs = 1.0f / sqrtf(ss / static_cast<float>(a.d) + a.eps);
            float z = 0.f;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float x = u[e] * rs + bd[e];
                z = fmaf(wu[e], __fdividef(x, 1.0f + __expf(-x)), z);   // SiLU (fast exp and divide: ~1e-6 relative)
            }
            z += __shfl_xor_sync(0xffffffffu, z, 1);
            z += __shfl_xor_sync(0xffffffffu, z, 2);
            z += __shfl_xor_sync(0xffffffffu, z, 4);
            const float p = __fdividef(1.0f, 1.0f + __expf(-(z + bu)));
            if (live) {
                if (cl == 0) {
                    a.score[t] = p;
                    if (a.rule == TEE_RULE_PER_TOKEN) a.mask[t] = exits(p, a.thr);
                }
                cmin = fminf(cmin, p == p ? p : -INFINITY);
            }
        }
        cmin = warp_min(cmin);
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 5) tc::tmem_dealloc(tmem, RBN);
    if (a.need_flag) flag_tail<RTHREADS>(cmin, a);
}

// ---- Large batches: a persistent CTA per SM (no cluster) takes whole token tiles
// in turn (tile = CTA + grid * i) over the whole d. Two 128-column TMEM
// accumulators: while warps 6-9 finish tile i straight from TMEM (thread = token:
// 1/rms, b_down, SiLU, w_up, sigmoid), warps 4 and 5 already stream and multiply
// tile i+1, and warps 0-3 sum its h^2. (Splitting the last tiles across CTAs, with
// the parts added through L2, was slower at every batch tried: the extra L2 round
// trips at the end cost more than the idle SMs of the last round.)
constexpr int PTHREADS = 10 * 32;
constexpr uint32_t PSMALL = 256 + 2 * RBM * 4 + 2 * RBN * 4;   // barriers | s_ss[2][128] | w_up, b_down
constexpr size_t PSMEM = 1024 + size_t(RSTAGES) * RSTAGE + PSMALL;

// The tiles of this CTA, walked alike by every role. Each tile's k stages are
// streamed from a CTA-dependent start (rot), wrapping, so that the CTAs do not all
// read the same W_down block from L2 at the same moment.
struct TileWalk {
    int tile, m_tiles, rot;
    __device__ __forceinline__ void begin(const RouterArgs& a) {
        m_tiles = (a.n + RBM - 1) / RBM;
        tile = static_cast<int>(blockIdx.x) - static_cast<int>(gridDim.x);
        rot = static_cast<int>(static_cast<int64_t>(blockIdx.x) * a.nks / gridDim.x);
    }
    __device__ __forceinline__ bool next() {
        tile += gridDim.x;
        return tile < m_tiles;
    }
};

__global__ void __launch_bounds__(PTHREADS, 1)
router_tc_persistent_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                            const __grid_constant__ RouterArgs a, void* ws) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + RSTAGES * RSTAGE);
    uint64_t* empty = full + RSTAGES;
    uint64_t* acc_full = empty + RSTAGES;   // [2] MMA commit: accumulator b holds a finished segment
    uint64_t* acc_empty = acc_full + 2;     // [2] the four epilogue warps are done with accumulator b
    uint64_t* ss_full = acc_empty + 2;      // [2] the four sum(h^2) warps wrote s_ss[b]
    uint64_t* mma_done = ss_full + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    float* s_ss = reinterpret_cast<float*>(smem + RSTAGES * RSTAGE + 256);   // [2][RBM]
    float* s_wu = s_ss + 2 * RBM;
    float* s_bd = s_wu + RBN;
    static_assert((2 * RSTAGES + 7) * 8 + 8 <= 256, "barrier block");

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    allow_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < RSTAGES; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1 + 4);   // MMA commit + the four sum(h^2) warps
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&acc_full[b], 1);
            tc::mbar_init(&acc_empty[b], 4);
            tc::mbar_init(&ss_full[b], 4);
        }
        tc::mbar_init(mma_done, 1);
        *abort = 0;
        tc::fence_barrier_init();
    }
    for (int c = threadIdx.x; c < RBN; c += PTHREADS) {
        s_wu[c] = __bfloat162float(a.w_up[c]);
        s_bd[c] = a.b_down ? a.b_down[c] : 0.f;
    }
    if (warp == 5) tc::tmem_alloc(tmem_slot, 2 * RBN);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    float cmin = INFINITY;
    TileWalk sw;
    sw.begin(a);

    if (warp == 4) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_phase = 0;
            bool ok = true;
            while (ok && sw.next()) {
                for (int i = 0; i < a.nks; ++i) {
                    const int kb = (i + sw.rot) % a.nks;
                    if (!tc::mbar_wait(&empty[stage], phase ^ 1, abort, ws, 41)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sa = smem + stage * RSTAGE;
                    tc::mbar_arrive_expect_tx(&full[stage], RSTAGE);
                    tc::tma_load_3d(sa, &tmA, 0, sw.tile * RBM, kb * RKZ, &full[stage]);
                    tc::tma_load_3d(sa + RA_STAGE, &tmB, 0, 0, kb * RKZ, &full[stage]);
                    issued |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == RSTAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (*abort) {   // let the copies already issued land before the block moves on
                for (int s = 0; s < RSTAGES; ++s) {
                    if (!(issued >> s & 1)) continue;
                    const uint64_t t0 = tc::globaltimer();
                    while (!tc::mbar_try_wait(&full[s], issued_phase >> s & 1) &&
                           tc::globaltimer() - t0 < tc::WAIT_LIMIT_NS) {
                    }
                }
            }
        }
    } else if (warp == 5) {
        if (lane == 0) {
            int stage = 0, it = 0;
            uint32_t phase = 0;
            constexpr uint32_t idesc = tc::idesc_bf16(RBM, RBN);
            bool ok = true;
            for (; ok && sw.next(); ++it) {
                const int b = it & 1;
                if (it >= 2 && !tc::mbar_wait(&acc_empty[b], ((it >> 1) - 1) & 1, abort, ws, 42)) break;
                tc::tc_fence_after();
                const uint32_t acc = tmem + b * RBN;
                for (int kb = 0; kb < a.nks; ++kb) {
                    if (!tc::mbar_wait(&full[stage], phase, abort, ws, 43)) {
                        ok = false;
                        break;
                    }
                    tc::tc_fence_after();
                    const uint32_t sa = tc::smem_u32(smem + stage * RSTAGE);
#pragma unroll
                    for (int z = 0; z < RKZ; ++z) {
                        const uint64_t ad = tc::smem_desc_sw128(sa + z * RA_BYTES);
                        const uint64_t bd = tc::smem_desc_sw128(sa + RA_STAGE + z * RB_BYTES);
#pragma unroll
                        for (int k = 0; k < RBK / 16; ++k)
                            tc::umma_bf16(acc, ad + 2 * k, bd + 2 * k, idesc, kb | z | k);
                    }
                    tc::umma_commit(&empty[stage]);
                    if (++stage == RSTAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (ok) tc::umma_commit(&acc_full[b]);
            }
            // Every MMA issued has finished before the accumulators are freed (also
            // after an abort: this wait ignores the flag and ends by its time limit).
            tc::umma_commit(mma_done);
            const uint64_t t0 = tc::globaltimer();
            while (!tc::mbar_try_wait(mma_done, 0) && tc::globaltimer() - t0 < tc::WAIT_LIMIT_NS) {
            }
        }
    } else if (warp < 4) {
        // sum(h^2) of token row (warp*32 + lane) over each segment's staged h tiles
        const int r = warp * 32 + lane;
        int stage = 0, it = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (; ok && sw.next(); ++it) {
            float ss = 0.f;
            for (int kb = 0; kb < a.nks; ++kb) {
                // every lane waits (each acquires the TMA writes); the outcome is made
                // warp-uniform so that a timeout cannot split the warp at __syncwarp
                if (!__all_sync(0xffffffffu, tc::mbar_wait(&full[stage], phase, abort, ws, 45))) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int jj = 0; jj < 8 * RKZ; ++jj) {
                    const int j = jj & 7;
                    const uint8_t* row = smem + stage * RSTAGE + (jj >> 3) * RA_BYTES + r * 128;
                    const uint4 v = *reinterpret_cast<const uint4*>(row + (((j + r) & 7) << 4));
                    float x[8];
                    unpack_bf16x2(v.x, x[0], x[1]);
                    unpack_bf16x2(v.y, x[2], x[3]);
                    unpack_bf16x2(v.z, x[4], x[5]);
                    unpack_bf16x2(v.w, x[6], x[7]);
#pragma unroll
                    for (int q = 0; q < 8; ++q) ss = fmaf(x[q], x[q], ss);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&empty[stage]);
                if (++stage == RSTAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (!ok) break;
            const int b = it & 1;
            // s_ss[b] is free once the epilogue of segment it - 2 has finished with it.
            if (it >= 2 && !__all_sync(0xffffffffu, tc::mbar_wait(&acc_empty[b], ((it >> 1) - 1) & 1, abort, ws, 46)))
                break;
            s_ss[b * RBM + r] = ss;
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&ss_full[b]);
        }
    } else {
        // warps 6-9: thread = token row q*32 + lane of the tile (TMEM lane quarter q = warp % 4)
        const int q = warp & 3, r = q * 32 + lane;
        const float bu = a.b_up ? a.b_up[0] : 0.f;
        const float inv_d = 1.0f / static_cast<float>(a.d);
        for (int it = 0; sw.next(); ++it) {
            const int b = it & 1;
            const uint32_t par = (it >> 1) & 1;
            bool ok = true;
            if (lane == 0)
                ok = tc::mbar_wait(&acc_full[b], par, abort, ws, 47) && tc::mbar_wait(&ss_full[b], par, abort, ws, 48);
            if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;   // warp-uniform: tcgen05.ld is collective
            __syncwarp();
            tc::tc_fence_after();
            const int t = sw.tile * RBM + r;
            const uint32_t tb = tmem + (static_cast<uint32_t>(q * 32) << 16) + b * RBN;
            const float rs = 1.0f / sqrtf(s_ss[b * RBM + r] * inv_d + a.eps);
            float z = 0.f;
#pragma unroll 1
            for (int c0 = 0; c0 < RBN; c0 += 32) {
                float v[32];
                tc::tmem_ld32(tb + c0, v);
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const float x = v[e] * rs + s_bd[c0 + e];
                    z = fmaf(s_wu[c0 + e], __fdividef(x, 1.0f + __expf(-x)), z);   // SiLU (fast exp and divide)
                }
            }
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&acc_empty[b]);
            if (t < a.n) {
                const float p = __fdividef(1.0f, 1.0f + __expf(-(z + bu)));
                a.score[t] = p;
                if (a.rule == TEE_RULE_PER_TOKEN) a.mask[t] = exits(p, a.thr);
                cmin = fminf(cmin, p == p ? p : -INFINITY);
            }
        }
        cmin = warp_min(cmin);
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 5) tc::tmem_dealloc(tmem, 2 * RBN);
    if (a.need_flag) flag_tail<PTHREADS>(cmin, a);
}

// K split: a power of two up to RMAX_SPLIT, about one wave of CTAs.
int router_splits(int n, int d) {
    const int m_tiles = (n + RBM - 1) / RBM, nks = (d / RBK + RKZ - 1) / RKZ;
    int s = 1;
    while (s * 2 <= RMAX_SPLIT && m_tiles * s * 2 <= sm_count() && s * 2 <= nks) s *= 2;
    return s;
}

}  // namespace

// Either grid is at most one CTA per SM, within the flag's 1024 per-CTA minima.
bool router_tc_eligible(int n, int d, int b, int dtype, const void* gamma) {
    return dtype == TEE_BF16 && b == RBN && !gamma && n >= RTC_MIN_TOKENS && d % RBK == 0;
}

// Scratch of a K split of `splits` (none without a split: the persistent kernel
// finishes its tiles from TMEM).
size_t router_tc_scratch_bytes_at(int n, int splits) {
    if (splits <= 1) return 0;
    const size_t rows = static_cast<size_t>((n + RBM - 1) / RBM) * splits * RBM;
    return round_up(rows * RBN * 4, 256) + round_up(rows * 4, 256);
}
// Scratch at the split the call prefers (the workspace size to ask for); a smaller
// workspace makes the call use a smaller split, down to router_tc_scratch_bytes_at(n, 1).
size_t router_tc_scratch_bytes(int n, int d, int b) {
    if (b != RBN || n < RTC_MIN_TOKENS || d % RBK) return 0;
    return router_tc_scratch_bytes_at(n, router_splits(n, d));
}

tee_status router_gate_tc(int n, int d, int b, int dtype, const void* h, int64_t ldh, const void* gamma,
                          const void* w_down, const float* b_down, const void* w_up, const float* b_up, float eps,
                          float thr, int rule, bool need_flag, float* score, uint8_t* mask, int32_t* flag,
                          float* block_mins, uint32_t* counter, void* ws, size_t ws_off, size_t ws_bytes,
                          cudaStream_t stream) {
    if (!router_tc_eligible(n, d, b, dtype, gamma)) return TEE_ERR_UNSUPPORTED;
    if ((ldh * 2) % 16 || !aligned16(h) || !aligned16(w_down) || (b_down && !aligned16(b_down)))
        return TEE_ERR_UNSUPPORTED;
    int splits = router_splits(n, d);
    while (splits > 1 && ws_off + router_tc_scratch_bytes_at(n, splits) > ws_bytes) splits >>= 1;
    if (ws_off + router_tc_scratch_bytes_at(n, splits) > ws_bytes) return TEE_ERR_WORKSPACE;
    CUtensorMap ta, tb;
    tee_status st = make_tmap_bf16_kblocks(&ta, h, n, static_cast<uint64_t>(ldh) * 2, d / RBK, RBM, RKZ);
    if (st != TEE_OK) return st == TEE_ERR_INVALID_ARG ? TEE_ERR_UNSUPPORTED : st;
    st = make_tmap_bf16_kblocks(&tb, w_down, RBN, static_cast<uint64_t>(d) * 2, d / RBK, RBN, RKZ);
    if (st != TEE_OK) return st == TEE_ERR_INVALID_ARG ? TEE_ERR_UNSUPPORTED : st;
    static bool attr = false;
    if (!attr) {
        st = cuda_status(cudaFuncSetAttribute(router_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              static_cast<int>(RSMEM)));
        if (st != TEE_OK) return st;
        st = cuda_status(cudaFuncSetAttribute(router_tc_persistent_kernel,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(PSMEM)));
        if (st != TEE_OK) return st;
        attr = true;
    }
    const int m_tiles = (n + RBM - 1) / RBM, nks = (d / RBK + RKZ - 1) / RKZ;
    RouterArgs a{};
    a.n = n;
    a.d = d;
    a.nks = nks;
    a.eps = eps;
    a.thr = thr;
    a.rule = rule;
    a.need_flag = need_flag;
    if (splits > 1) {
        char* p = static_cast<char*>(ws) + ws_off;
        const size_t rows = static_cast<size_t>(m_tiles) * splits * RBM;
        a.part = reinterpret_cast<float*>(p);
        a.part_ss = reinterpret_cast<float*>(p + round_up(rows * RBN * 4, 256));
    }
    a.b_down = b_down;
    a.w_up = static_cast<const bf16*>(w_up);
    a.b_up = b_up;
    a.score = score;
    a.mask = mask;
    a.flag = flag;
    a.block_mins = block_mins;
    a.counter = counter;

    if (splits == 1) {   // persistent: one CTA per SM over the token tiles
        const int grid = m_tiles < sm_count() ? m_tiles : sm_count();
        router_tc_persistent_kernel<<<grid, PTHREADS, PSMEM, stream>>>(ta, tb, a, ws);
        return launch_status();
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(m_tiles, splits);
    cfg.blockDim = dim3(RTHREADS);
    cfg.dynamicSmemBytes = RSMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attrs[1];
    attrs[0].id = cudaLaunchAttributeClusterDimension;
    attrs[0].val.clusterDim.x = 1;
    attrs[0].val.clusterDim.y = splits;
    attrs[0].val.clusterDim.z = 1;
    cfg.attrs = attrs;
    cfg.numAttrs = 1;
    st = cuda_status(cudaLaunchKernelEx(&cfg, router_tc_kernel, ta, tb, a, ws));
    return st != TEE_OK ? st : launch_status();
}

}  // namespace tee
