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

constexpr int RBM = 128, RBN = 128, RBK = 64, RSTAGES = 6;
constexpr int RTHREADS = 6 * 32;
constexpr int RMAX_SPLIT = 4;   // K split and cluster size at most (keeps the finishing loads in registers)
constexpr uint32_t RA_BYTES = RBM * RBK * 2, RB_BYTES = RBN * RBK * 2, RSTAGE = RA_BYTES + RB_BYTES;
constexpr int RSTAGE_LD = 132;  // floats per staged row (conflict-free 16-byte stores)
constexpr uint32_t RSTAGING = 4 * 32 * RSTAGE_LD * 4;   // epilogue staging: reuses the ring once the MMAs are done
static_assert(RSTAGING <= RSTAGES * RSTAGE, "staging must fit in the ring");
constexpr size_t RSMEM = 1024 + size_t(RSTAGES) * RSTAGE + 256;
// Smallest batch that goes to the tensor cores.
constexpr int RTC_MIN_TOKENS = 256;

struct RouterArgs {
    int n, d, nkb, kbps;
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
    const int kb0 = split * a.kbps;
    const int kb1 = min(kb0 + a.kbps, a.nkb);
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
                tc::tma_load_2d(sa, &tmA, kb * RBK, m0, &full[stage]);
                tc::tma_load_2d(sa + RA_BYTES, &tmB, kb * RBK, 0, &full[stage]);
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
                const uint64_t ad = tc::smem_desc_sw128(sa), bd = tc::smem_desc_sw128(sa + RA_BYTES);
#pragma unroll
                for (int k = 0; k < RBK / 16; ++k) tc::umma_bf16(tmem, ad + 2 * k, bd + 2 * k, idesc, (kb - kb0) | k);
                tc::umma_commit(&empty[stage]);
                if (++stage == RSTAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            tc::umma_commit(acc_full);  // also when stopped early: every issued MMA finishes first
        }
    } else {
        // warps 0-3: sum(h^2) of token row (warp*32 + lane) from each staged h tile
        const int r = warp * 32 + lane;
        float ss = 0.f;
        int stage = 0;
        uint32_t phase = 0;
        for (int kb = kb0; kb < kb1; ++kb) {
            if (!tc::mbar_wait(&full[stage], phase, abort, ws, 33)) {
                ok = false;
                break;
            }
            const uint8_t* row = smem + stage * RSTAGE + r * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                // rotate the chunk order by row: lanes of a warp hit 8 different bank groups
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
    if (!a.need_flag) return;
    // All-tokens flag: each CTA publishes its minimum; the last CTA to arrive reduces.
    __shared__ float s_min[RTHREADS / 32];
    if (lane == 0) s_min[warp] = cmin;
    __syncthreads();
    __shared__ int s_last;
    const int nblocks = gridDim.x * gridDim.y, bid = blockIdx.y * gridDim.x + blockIdx.x;
    if (threadIdx.x == 0) {
        float m = INFINITY;
        for (int w = 0; w < RTHREADS / 32; ++w) m = fminf(m, s_min[w]);
        a.block_mins[bid] = m;
        __threadfence();
        s_last = atomicAdd(a.counter, 1u) == static_cast<unsigned>(nblocks - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    float m = INFINITY;
    for (int i = threadIdx.x; i < nblocks; i += RTHREADS) m = fminf(m, *reinterpret_cast<volatile float*>(a.block_mins + i));
    m = warp_min(m);
    if (lane == 0) s_min[warp] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float mm = INFINITY;
        for (int w = 0; w < RTHREADS / 32; ++w) mm = fminf(mm, s_min[w]);
        s_min[0] = mm;
    }
    __syncthreads();
    const uint8_t f = (a.n > 0 && s_min[0] > a.thr) ? 1 : 0;
    if (threadIdx.x == 0) {
        if (a.flag) *a.flag = f;
        *a.counter = 0u;
    }
    if (a.rule == TEE_RULE_BATCH_ALL)
        for (int t = threadIdx.x; t < a.n; t += RTHREADS) a.mask[t] = f;
}

// K split: a power of two up to RMAX_SPLIT, about one wave of CTAs.
int router_splits(int n, int d) {
    const int m_tiles = (n + RBM - 1) / RBM, nkb = d / RBK;
    int s = 1;
    while (s * 2 <= RMAX_SPLIT && m_tiles * s * 2 <= sm_count() && s * 2 <= nkb) s *= 2;
    return s;
}

}  // namespace

bool router_tc_eligible(int n, int d, int b, int dtype, const void* gamma) {
    return dtype == TEE_BF16 && b == RBN && !gamma && n >= RTC_MIN_TOKENS && d % RBK == 0 &&
           (n + RBM - 1) / RBM * router_splits(n, d) <= 1024;   // the flag's per-CTA minima
}

size_t router_tc_scratch_bytes_at(int n, int splits) {
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
    tee_status st = make_tmap_bf16(&ta, h, d, n, static_cast<uint64_t>(ldh) * 2, RBK, RBM);
    if (st != TEE_OK) return st == TEE_ERR_INVALID_ARG ? TEE_ERR_UNSUPPORTED : st;
    st = make_tmap_bf16(&tb, w_down, d, RBN, static_cast<uint64_t>(d) * 2, RBK, RBN);
    if (st != TEE_OK) return st == TEE_ERR_INVALID_ARG ? TEE_ERR_UNSUPPORTED : st;
    static bool attr = false;
    if (!attr) {
        st = cuda_status(cudaFuncSetAttribute(router_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              static_cast<int>(RSMEM)));
        if (st != TEE_OK) return st;
        attr = true;
    }
    const int m_tiles = (n + RBM - 1) / RBM, nkb = d / RBK;
    RouterArgs a{};
    a.n = n;
    a.d = d;
    a.nkb = nkb;
    a.kbps = (nkb + splits - 1) / splits;
    a.eps = eps;
    a.thr = thr;
    a.rule = rule;
    a.need_flag = need_flag;
    char* p = static_cast<char*>(ws) + ws_off;
    const size_t rows = static_cast<size_t>(m_tiles) * splits * RBM;
    a.part = reinterpret_cast<float*>(p);
    a.part_ss = reinterpret_cast<float*>(p + round_up(rows * RBN * 4, 256));
    a.b_down = b_down;
    a.w_up = static_cast<const bf16*>(w_up);
    a.b_up = b_up;
    a.score = score;
    a.mask = mask;
    a.flag = flag;
    a.block_mins = block_mins;
    a.counter = counter;

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
