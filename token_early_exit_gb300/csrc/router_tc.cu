// TIDE router contraction on tcgen05 for large batches (formula 3; module 4
// "Fused LayerNorm + Route"): dots[t][c] = sum_i W_down[c][i] h[t][i] and
// sumsq[t] = sum_i h[t][i]^2, the inputs of the router's finalize kernel
// (1/rms, b_down, SiLU, w_up, sigmoid, threshold).
//
// M = 128 tokens, N = 128 router channels, K = d split across CTAs so that a
// 4096-token batch spreads over ~128 SMs. W_down [128][d] is already K-major,
// so TMA reads the caller's weights directly. Warp 4 streams 128x64 tiles of h
// and W_down into a 4-stage ring (128-byte swizzle), one thread of warp 5
// issues tcgen05.mma into a 128-column TMEM accumulator, and warps 0-3 add up
// sum(h^2) of their token row from each staged h tile (a ring slot is freed by
// the MMA commit plus the four warps). At the end each of warps 0-3 reads its
// 32 token rows from TMEM and adds them into dots with vector reductions; the
// finalize kernel clears dots and sumsq after reading them.
#include "tc.cuh"

namespace tee {

namespace {

using bf16 = __nv_bfloat16;

constexpr int RBM = 128, RBN = 128, RBK = 64, RSTAGES = 4;
constexpr int RTHREADS = 6 * 32;
constexpr uint32_t RA_BYTES = RBM * RBK * 2, RB_BYTES = RBN * RBK * 2, RSTAGE = RA_BYTES + RB_BYTES;
constexpr int RSTAGE_LD = 132;  // floats per staged row (conflict-free 16-byte stores)
constexpr uint32_t RSTAGING = 4 * 32 * RSTAGE_LD * 4;   // epilogue staging, its own region
constexpr size_t RSMEM = 1024 + size_t(RSTAGES) * RSTAGE + RSTAGING + 256;
// Smallest batch that goes to the tensor cores.
constexpr int RTC_MIN_TOKENS = 256;

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

__global__ void __launch_bounds__(RTHREADS, 1)
router_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, int n, int nkb,
                 int kb_per_split, float* __restrict__ dots, float* __restrict__ sumsq, void* ws) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* staging = reinterpret_cast<float*>(smem + RSTAGES * RSTAGE);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + RSTAGES * RSTAGE + RSTAGING);
    uint64_t* empty = full + RSTAGES;
    uint64_t* acc_full = empty + RSTAGES;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * RBM;
    const int kb0 = blockIdx.y * kb_per_split;
    const int kb1 = min(kb0 + kb_per_split, nkb);

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
            if (*abort) {
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
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!tc::mbar_wait(&full[stage], phase, abort, ws, 32)) {
                    ok = false;
                    break;
                }
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
            (void)ok;
            tc::umma_commit(acc_full);  // also when stopped early: every issued MMA finishes first
        }
    } else {
        // warps 0-3: sum(h^2) of token row (warp*32 + lane) from each staged h tile
        const int r = warp * 32 + lane;
        float ss = 0.f;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
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
        const int t = m0 + r;
        if (ok) {
            // Stage this warp's 32 rows in shared memory (row stride 132 floats keeps
            // the 16-byte stores conflict-free), then add each row into dots with
            // one 512-byte vector reduction per warp instruction.
            float* stage = staging + warp * (32 * RSTAGE_LD);
            const uint32_t tb = tmem + (static_cast<uint32_t>(warp * 32) << 16);
#pragma unroll 1
            for (int c = 0; c < RBN; c += 32) {
                float v[32];
                tc::tmem_ld32(tb + c, v);
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    *reinterpret_cast<float4*>(stage + lane * RSTAGE_LD + c + 4 * q) =
                        make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            }
            __syncwarp();
            for (int rr = 0; rr < 32; ++rr) {
                const int tt = m0 + warp * 32 + rr;
                if (tt >= n) break;
                const float4 v = *reinterpret_cast<const float4*>(stage + rr * RSTAGE_LD + lane * 4);
                red_add_v4(dots + static_cast<int64_t>(tt) * RBN + lane * 4, v.x, v.y, v.z, v.w);
            }
            if (t < n) atomicAdd(sumsq + t, ss);
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 5) tc::tmem_dealloc(tmem, RBN);
}

}  // namespace

size_t router_tc_scratch_bytes(int n, int d, int b) {
    (void)n;
    (void)d;
    (void)b;
    return 0;  // accumulates into the dots / sumsq area the CUDA-core path uses
}

tee_status router_dots_tc(int n, int d, int b, int dtype, const void* h, int64_t ldh, const void* gamma,
                          const void* w_down, float* dots, float* sumsq, void* ws, size_t ws_off, size_t ws_bytes,
                          cudaStream_t stream) {
    (void)ws_off;
    (void)ws_bytes;
    if (dtype != TEE_BF16 || b != RBN || gamma || n < RTC_MIN_TOKENS || d % RBK) return TEE_ERR_UNSUPPORTED;
    if ((ldh * 2) % 16 || !aligned16(h) || !aligned16(w_down)) return TEE_ERR_UNSUPPORTED;
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
    // One wave: m_tiles * splits <= SMs (a second partial wave doubles the time).
    int splits = sm_count() / m_tiles;
    if (splits > nkb) splits = nkb;
    if (splits > 16) splits = 16;
    if (splits < 1) splits = 1;
    const int kbps = (nkb + splits - 1) / splits;
    splits = (nkb + kbps - 1) / kbps;
    router_tc_kernel<<<dim3(m_tiles, splits), RTHREADS, RSMEM, stream>>>(ta, tb, n, nkb, kbps, dots, sumsq, ws);
    return launch_status();
}

}  // namespace tee
