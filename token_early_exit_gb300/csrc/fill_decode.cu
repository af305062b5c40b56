// Decode path of the KV fill: up to 128 items (decode tokens that exit), int4
// group-64 weights (River-LLM's W4A16 exit layers), identity map (the
// "State Propagation" / identity-fill input).
//
// One launch, one CTA per (group of 64 output columns, filled layer). The 64
// columns are two 32-wide segments [i, i+32) and [i+hd/2, i+hd/2+32) of one K
// or V head, so that RoPE pairs stay inside the CTA. On tcgen05:
//   D[item][c] = sum_k h[row(item)][k] * W'[k][c],  M = 128 item rows (rows
//   past the items hold whatever; their D rows are never stored), N = 64
//   columns, K = d, with
//   W'[k][c] = (q - zero) * scale * g_j[k]
// so that D / rms(h) is layer j's K or V for each item (RMSNorm weight folded
// into the dequantised weights). Warp roles, synchronised by mbarriers only:
//   warps 0-7   stream the int4 codes, fp16 scales/zeros and g_j in 512-k
//               chunks (cp.async, a 3-chunk ring) and dequantise each 64-k
//               block into a ring of bf16 B operands (128-byte swizzle);
//   warp 8      issues tcgen05.mma into a 64-column TMEM accumulator and frees
//               the ring slots with tcgen05.commit;
//   warps 9-12  gather the items' h rows of each 64-k block into a ring of A
//               operands (cp.async, 128-byte swizzle), two blocks in flight,
//               after asking L2 for the whole rows at the start; once a
//               thread's copies of a block have landed it fences them for the
//               tensor core and releases the block. They also fetch the
//               items' positions, cache slots and RoPE rows;
//   warps 13-14 add up sum(h^2) per item from each landed A block.
// Epilogue (warps 0-3, one item row each): 1/rms, RoPE in registers, store of
// the two 32-wide segments into the backbone's cache slot.
#include "fill.cuh"
#include "tc.cuh"

namespace tee {

namespace {

using bf16 = __nv_bfloat16;

constexpr int D_COLS = 64;           // output columns per CTA
constexpr int D_KB = 64;             // K per MMA block (one int4 group)
constexpr int D_CHUNK = 512;         // K per staged chunk of codes
constexpr int D_RA = 6;              // A operand slots (h rows)
constexpr int D_LAG = 2;             // blocks of h copies in flight
constexpr int D_RB = 3;              // B operand slots (dequantised weights)
constexpr int D_RC = 3;              // code chunks in the ring
constexpr int D_MAX_ITEMS = 128;
constexpr int D_DEQ_WARPS = 8, D_MMA_WARP = 8, D_CP_WARP0 = 9, D_CP_WARPS = 4, D_SS_WARP0 = 13, D_SS_WARPS = 2;
constexpr int D_CP_THREADS = D_CP_WARPS * 32;
constexpr int D_ITEMS_PER_CP = D_MAX_ITEMS * 8 / D_CP_THREADS;   // 16-byte pieces per thread and block
constexpr int D_THREADS = (D_SS_WARP0 + D_SS_WARPS) * 32;
constexpr int D_CROW = D_COLS + 16;  // staged bytes per packed-code row (padding spreads the banks)
// A slot is refilled D_RA - D_LAG - 1 iterations after its release: slack for the MMA
// and sum(h^2) round trip (mbarrier hand-offs cost ~0.1 us each).
static_assert(D_LAG + 2 < D_RA, "the A ring needs slack beyond the blocks in flight");

constexpr uint32_t A_SLOT = 128 * 128;                                   // 16 KB
constexpr uint32_t B_SLOT = D_COLS * 128;                                // 8 KB
constexpr uint32_t CHUNK_CODES = (D_CHUNK / 2) * D_CROW;                 // 20 KB
constexpr uint32_t CHUNK_SZ = (D_CHUNK / D_KB) * 256;                    // scale[64], zero[64] per group: 2 KB
constexpr uint32_t CHUNK_G = D_CHUNK * 2;                                // 1 KB
constexpr uint32_t CHUNK_BYTES = CHUNK_CODES + CHUNK_SZ + CHUNK_G;
constexpr uint32_t OFF_A = 0;
constexpr uint32_t OFF_B = OFF_A + D_RA * A_SLOT;
constexpr uint32_t OFF_C = OFF_B + D_RB * B_SLOT;
constexpr uint32_t OFF_ROPE = OFF_C + D_RC * CHUNK_BYTES;                // float2 [item][32]
constexpr uint32_t OFF_SMALL = OFF_ROPE + D_MAX_ITEMS * 256;
constexpr uint32_t SMALL_BYTES = (2 * D_RA + 2 * D_RB + 2) * 8 + D_MAX_ITEMS * (8 + 4) + 16;
constexpr size_t D_SMEM = 1024 + OFF_SMALL + SMALL_BYTES;
static_assert(D_SMEM <= 232448, "decode fill shared memory");
static_assert(OFF_B % 1024 == 0 && OFF_C % 16 == 0 && OFF_ROPE % 16 == 0 && OFF_SMALL % 8 == 0, "alignment");

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
    int n_max, d, kvw, hd, half, n_kv, groups_per_head;
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
    asm volatile("bar.sync 1, %0;" ::"n"(D_DEQ_WARPS * 32) : "memory");
}
__device__ __forceinline__ float nibble_f32(uint32_t q) {
    // exact small integer as fp32: (2^23 + q) - 2^23
    return __uint_as_float(0x4B000000u | q) - 8388608.0f;
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
    int64_t* s_off = reinterpret_cast<int64_t*>(ss_ready + 1);        // cache offset of the item row or -1
    float* s_ss = reinterpret_cast<float*>(s_off + D_MAX_ITEMS);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s_ss + D_MAX_ITEMS);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int grp = blockIdx.x, li = blockIdx.y;
    const DecodeLayer& L = a.l[li];
    const bool is_k = grp < a.n_kv * a.groups_per_head;
    const int kv = is_k ? 0 : 1;
    const int gi = is_k ? grp : grp - a.n_kv * a.groups_per_head;
    const int head = gi / a.groups_per_head, seg = gi % a.groups_per_head;
    const int col_lo = head * a.hd + 32 * seg, col_hi = col_lo + a.half;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nkb = a.d / D_KB, nchunks = a.d / D_CHUNK;
    const bool reporter = grp == 0 && li == 0;   // one block records bad rows / positions

    if (threadIdx.x == 0) {
        for (int s = 0; s < D_RA; ++s) {
            tc::mbar_init(&a_full[s], D_CP_WARPS);
            tc::mbar_init(&a_empty[s], 1 + D_SS_WARPS);   // MMA commit + the sum(h^2) warps
        }
        for (int s = 0; s < D_RB; ++s) {
            tc::mbar_init(&b_full[s], D_DEQ_WARPS);
            tc::mbar_init(&b_empty[s], 1);
        }
        tc::mbar_init(acc_full, 1);
        tc::mbar_init(ss_ready, D_CP_WARPS + D_SS_WARPS);
        *abort = 0;
        tc::fence_barrier_init();
    }
    // Chunk c of codes / scales / zeros / g into ring slot c % D_RC (dequant warps).
    auto load_chunk = [&](int c) {
        uint8_t* base = smem + OFF_C + (c % D_RC) * CHUNK_BYTES;
        const int kp0 = c * (D_CHUNK / 2), g0 = c * (D_CHUNK / D_KB);
        for (int u = threadIdx.x; u < (D_CHUNK / 2) * 4; u += D_DEQ_WARPS * 32) {
            const int r = u >> 2, part = u & 3;        // packed row, 16-byte piece (lo 2, hi 2)
            const int col = (part < 2 ? col_lo : col_hi) + (part & 1) * 16;
            cp_async16(base + r * D_CROW + part * 16, L.codes[kv] + static_cast<int64_t>(kp0 + r) * a.kvw + col);
        }
        for (int u = threadIdx.x; u < (D_CHUNK / D_KB) * 16 + D_CHUNK / 8; u += D_DEQ_WARPS * 32) {
            if (u < (D_CHUNK / D_KB) * 16) {
                const int g = u >> 4, part = u & 15, which = part >> 3, p = part & 7;
                const int col = (p < 4 ? col_lo : col_hi) + (p & 3) * 8;
                const __half* src = (which ? L.zero[kv] : L.scale[kv]) + static_cast<int64_t>(g0 + g) * a.kvw + col;
                cp_async16(base + CHUNK_CODES + g * 256 + which * 128 + p * 16, src);
            } else {
                const int p = u - (D_CHUNK / D_KB) * 16;
                cp_async16(base + CHUNK_CODES + CHUNK_SZ + p * 16, L.gamma + c * D_CHUNK + p * 8);
            }
        }
    };
    if (warp < D_DEQ_WARPS) {
        for (int c = 0; c < D_RC; ++c) {
            if (c < nchunks) load_chunk(c);
            cp_async_commit();
        }
    }
    if (warp == D_MMA_WARP) tc::tmem_alloc(tmem_slot, D_COLS);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < D_DEQ_WARPS) {
        // ---- dequantise: unit = 4 columns x 4 k, 256 units per 64-k block
        const int v = threadIdx.x;
        const int cg = ((v >> 5) & 3) * 4 + (v & 3);              // column group (4 columns)
        const int kq = (v >> 7) * 8 + ((v >> 2) & 7);             // k quad: 4kq .. 4kq+3
        bool ok = true;
        // Every dequantising warp runs every chunk iteration (the named barriers must
        // match); after a timed-out wait a warp only skips the work.
        for (int c = 0; c < nchunks; ++c) {
            cp_async_wait<D_RC - 1>();                            // chunk c has landed (own copies)
            deq_bar_sync();                                       // ... and everyone's
            const uint8_t* base = smem + OFF_C + (c % D_RC) * CHUNK_BYTES;
            for (int b = 0; b < D_CHUNK / D_KB && ok; ++b) {
                const int kb = c * (D_CHUNK / D_KB) + b, s = kb % D_RB;
                if (kb >= D_RB && !warp_wait(&b_empty[s], ((kb / D_RB) - 1) & 1, abort, ws, 51)) {
                    ok = false;
                    break;
                }
                const uint8_t* crow = base + (b * 32 + 2 * kq) * D_CROW + 4 * cg;
                const uint32_t w0 = *reinterpret_cast<const uint32_t*>(crow);
                const uint32_t w1 = *reinterpret_cast<const uint32_t*>(crow + D_CROW);
                const uint8_t* szp = base + CHUNK_CODES + b * 256;
                const uint2 s4 = *reinterpret_cast<const uint2*>(szp + cg * 8);
                const uint2 z4 = *reinterpret_cast<const uint2*>(szp + 128 + cg * 8);
                const uint2 g4 = *reinterpret_cast<const uint2*>(base + CHUNK_CODES + CHUNK_SZ + (b * D_KB + 4 * kq) * 2);
                float sc[4], zs[4], g[4];
                unpack_f16x2(s4.x, sc[0], sc[1]);
                unpack_f16x2(s4.y, sc[2], sc[3]);
                unpack_f16x2(z4.x, zs[0], zs[1]);
                unpack_f16x2(z4.y, zs[2], zs[3]);
                unpack_bf16x2(g4.x, g[0], g[1]);
                unpack_bf16x2(g4.y, g[2], g[3]);
                uint8_t* bslot = smem + OFF_B + s * B_SLOT;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float szj = zs[j] * sc[j];
                    const uint32_t b0 = (w0 >> (8 * j)) & 0xFFu, b1 = (w1 >> (8 * j)) & 0xFFu;
                    // (q - z) * s * g  as  (q * s - z * s) * g
                    const float x0 = fmaf(nibble_f32(b0 & 0xFu), sc[j], -szj) * g[0];
                    const float x1 = fmaf(nibble_f32(b0 >> 4), sc[j], -szj) * g[1];
                    const float x2 = fmaf(nibble_f32(b1 & 0xFu), sc[j], -szj) * g[2];
                    const float x3 = fmaf(nibble_f32(b1 >> 4), sc[j], -szj) * g[3];
                    const int col = 4 * cg + j, kc = kq >> 1;
                    *reinterpret_cast<uint2*>(bslot + col * 128 + ((kc ^ (col & 7)) << 4) + ((kq & 1) << 3)) =
                        make_uint2(pack_bf16x2(x0, x1), pack_bf16x2(x2, x3));
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&b_full[s]);
            }
            deq_bar_sync();                                       // everyone is done with chunk c
            if (c + D_RC < nchunks) load_chunk(c + D_RC);
            cp_async_commit();
        }
    } else if (warp == D_MMA_WARP) {
        // ---- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_bf16(128, D_COLS);
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
    } else if (warp < D_SS_WARP0) {
        // ---- h rows. Thread ct copies 16-byte piece j = ct % 8 of items ct / 8 + 16 m,
        // m = 0..7, of every block.
        const int ct = threadIdx.x - D_CP_WARP0 * 32;
        const int j = ct & 7, ib = ct >> 3;
        const int n = min(item_count(a.n_max, a.n_dev), D_MAX_ITEMS);
        // Item ct's h row, pulled into L2 whole (every block of it is read by every CTA).
        int r_ct = -1;
        if (ct < n) {
            const int r = a.rows ? a.rows[ct] : ct;
            if (r >= 0 && r < a.h_rows) {
                r_ct = r;
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a.h + static_cast<int64_t>(r) * a.ld_h),
                             "r"(a.d * 2)
                             : "memory");
            } else if (reporter) {
                record_fault(ws, TEE_DEVERR_ROW, r);
            }
        }
        const bf16* src[D_ITEMS_PER_CP];
#pragma unroll
        for (int m = 0; m < D_ITEMS_PER_CP; ++m) {
            const int i = ib + 16 * m;
            const int r = i < n ? (a.rows ? a.rows[i] : i) : -1;
            src[m] = (r >= 0 && r < a.h_rows) ? a.h + static_cast<int64_t>(r) * a.ld_h + j * 8 : nullptr;
        }
        auto issue = [&](int kb) {
            uint8_t* slot = smem + OFF_A + (kb % D_RA) * A_SLOT;
#pragma unroll
            for (int m = 0; m < D_ITEMS_PER_CP; ++m) {
                const int i = ib + 16 * m;
                if (src[m]) cp_async16(slot + i * 128 + ((j ^ (i & 7)) << 4), src[m] + kb * D_KB);
            }
        };
        // Block kb's copies (and all older ones) of this thread have landed: order them
        // for the tensor core and release the block.
        auto release = [&](int kb) {
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
            if (kb == 0) {
                // Item ct's position, cache slot and RoPE row (the RoPE copies ride in block 0's group).
                int64_t off = -1;
                if (r_ct >= 0) {
                    const int p = a.pos ? a.pos[r_ct] : a.pos0 + r_ct;
                    const int sq = a.seq ? a.seq[r_ct] : 0;
                    if (!pos_ok(p, a.cl.max_pos, a.hdr)) {
                        if (reporter) record_fault(ws, TEE_DEVERR_POS, p);
                    } else if (sq < 0 || sq >= a.cl.n_seq) {
                        if (reporter) record_fault(ws, TEE_DEVERR_SEQ, sq);
                    } else {
                        off = L.cache_layer * a.cl.s_layer + sq * a.cl.s_seq + head * a.cl.s_head +
                              static_cast<int64_t>(p) * a.cl.s_pos;
                        if (is_k)
                            for (int u = 0; u < 16; ++u)
                                cp_async16(smem + OFF_ROPE + ct * 256 + u * 16,
                                           a.rope + static_cast<int64_t>(p) * a.half + 32 * seg + u * 2);
                    }
                }
                s_off[ct] = off;
            }
            cp_async_commit();
            if (kb >= D_LAG) {
                cp_async_wait<D_LAG>();
                release(kb - D_LAG);
            }
        }
        cp_async_wait<0>();
        if (ok)
            for (int b = max(0, nkb - D_LAG); b < nkb; ++b) release(b);
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(ss_ready);   // release: s_off and the RoPE rows are ready
    } else {
        // ---- sum(h^2): warp w takes items 32 (2q + w) + lane, q = 0, 1, from each landed block.
        const int w = warp - D_SS_WARP0;
        const int n = min(item_count(a.n_max, a.n_dev), D_MAX_ITEMS);
        float ss[2] = {0.f, 0.f};
        for (int kb = 0; kb < nkb; ++kb) {
            const int s = kb % D_RA;
            if (!warp_wait(&a_full[s], (kb / D_RA) & 1, abort, ws, 55)) break;
            const uint8_t* slot = smem + OFF_A + s * A_SLOT;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int i = 32 * (2 * q + w) + lane;
                if (i >= n) continue;
#pragma unroll
                for (int jj = 0; jj < 8; ++jj)   // chunk order rotated by row: conflict-free across the warp
                    ss[q] = sumsq8(*reinterpret_cast<const uint4*>(slot + i * 128 + (((jj + i) & 7) << 4)), ss[q]);
            }
            // Order these reads before the refill of the slot.
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&a_empty[s]);
        }
#pragma unroll
        for (int q = 0; q < 2; ++q) s_ss[32 * (2 * q + w) + lane] = ss[q];
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(ss_ready);   // release: s_ss is ready
    }

    // ---- epilogue: warps 0-3, thread = item row = TMEM lane
    if (warp < 4) {
        bool ok = warp_wait(acc_full, 0, abort, ws, 56);
        ok = ok && warp_wait(ss_ready, 0, abort, ws, 57);
        tc::tc_fence_after();
        const int i = warp * 32 + lane;
        const int n = min(item_count(a.n_max, a.n_dev), D_MAX_ITEMS);
        const bool valid = ok && i < n && s_off[i] >= 0;
        const uint32_t tb = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        float lo[32], hi[32];
        tc::tmem_ld32(tb, lo);
        tc::tmem_ld32(tb + 32, hi);
        if (valid) {
            const float rs = 1.0f / sqrtf(s_ss[i] * a.inv_d + a.eps);
            if (is_k) {
                const float2* cs = reinterpret_cast<const float2*>(smem + OFF_ROPE + i * 256);
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const float2 e = cs[c];
                    const float x1 = lo[c] * rs, x2 = hi[c] * rs;
                    lo[c] = x1 * e.x - x2 * e.y;
                    hi[c] = x2 * e.x + x1 * e.y;
                }
            } else {
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    lo[c] *= rs;
                    hi[c] *= rs;
                }
            }
            bf16* dst = (is_k ? a.kc : a.vc) + s_off[i] + 32 * seg;
            uint4* o = reinterpret_cast<uint4*>(dst);
            uint4* o2 = reinterpret_cast<uint4*>(dst + a.half);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                o[q] = make_uint4(pack_bf16x2(lo[8 * q], lo[8 * q + 1]), pack_bf16x2(lo[8 * q + 2], lo[8 * q + 3]),
                                  pack_bf16x2(lo[8 * q + 4], lo[8 * q + 5]), pack_bf16x2(lo[8 * q + 6], lo[8 * q + 7]));
                o2[q] = make_uint4(pack_bf16x2(hi[8 * q], hi[8 * q + 1]), pack_bf16x2(hi[8 * q + 2], hi[8 * q + 3]),
                                   pack_bf16x2(hi[8 * q + 4], hi[8 * q + 5]), pack_bf16x2(hi[8 * q + 6], hi[8 * q + 7]));
            }
        }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == D_MMA_WARP) tc::tmem_dealloc(tmem, D_COLS);
}

bool decode_eligible(const FillCall& fc) {
    const tee_fill_desc& D = *fc.desc;
    if (D.dtype != TEE_BF16 || D.wfmt != TEE_W_INT4 || D.group != D_KB) return false;
    if (fc.n_max > D_MAX_ITEMS || fc.n_layers > MAX_DECODE_LAYERS) return false;
    if (D.d % D_CHUNK || (D.head_dim != 64 && D.head_dim != 128)) return false;
    if ((fc.ld_h * 2) % 16 || !aligned16(fc.h) || !aligned16(fc.k_cache) || !aligned16(fc.v_cache)) return false;
    const tee_cache_layout& cl = *fc.cache;
    if (cl.s_layer % 8 || cl.s_seq % 8 || cl.s_head % 8 || cl.s_pos % 8) return false;
    const int kvw = D.n_kv_heads * D.head_dim;
    if (kvw % 16) return false;
    for (int l = 0; l < fc.n_layers; ++l) {
        const tee_fill_layer& L = fc.layers[l];
        if (L.w_map) return false;
        if (!aligned16(L.wk) || !aligned16(L.wv) || !aligned16(L.k_scale) || !aligned16(L.k_zero) ||
            !aligned16(L.v_scale) || !aligned16(L.v_zero) || !aligned16(L.gamma))
            return false;
    }
    return true;
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
    DecodeArgs a{};
    a.n_max = fc.n_max;
    a.n_dev = fc.n_dev;
    a.d = D.d;
    a.kvw = D.n_kv_heads * D.head_dim;
    a.hd = D.head_dim;
    a.half = D.head_dim / 2;
    a.n_kv = D.n_kv_heads;
    a.groups_per_head = a.half / 32;
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
    static bool attr = false;
    if (!attr) {
        tee_status st = cuda_status(cudaFuncSetAttribute(fill_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                         static_cast<int>(D_SMEM)));
        if (st != TEE_OK) return st;
        attr = true;
    }
    dim3 grid(2 * a.n_kv * a.groups_per_head, fc.n_layers);
    fill_decode_kernel<<<grid, D_THREADS, D_SMEM, fc.stream>>>(a, fc.ws);
    return launch_status();
}

}  // namespace tee
