// Decode path of the KV fill: up to 128 items (decode tokens that exit), int4
// group-64 weights (River-LLM's W4A16 exit layers), identity map (the
// "State Propagation" / identity-fill input).
//
// One launch, one CTA per (head of K or V, filled layer). On tcgen05:
//   D[item][c] = sum_k h[row(item)][k] * W'[k][c],  M = 128 item rows,
//   N = head_dim columns, K = d,   W'[k][c] = (q - zero) * scale * g_j[k]
// so that D / rms(h) is layer j's K (or V) head for each item; the RMSNorm
// weight g_j is folded into the dequantised weights.
//
// Shared memory holds an 8-slot ring of raw inputs per 64-wide K block, filled
// six blocks ahead with cp.async: the gathered h rows land directly in the
// 128-byte-swizzled K-major A operand layout (rows past the items read as
// zero), next to the block's int4 codes, fp16 scales/zeros and g_j. Per block,
// warps 0-3 dequantise the codes into the B operand (bf16, swizzled, double
// buffered) while warps 4-7 add up sum(h^2) of their item row from the staged
// A tile; one thread then issues four tcgen05.mma (K = 16) and commits to the
// slot's barrier, which frees both the slot and the B buffer. After the last
// block each epilogue thread owns one item row of the TMEM accumulator, i.e. a
// whole head: it applies 1/rms and RoPE (pairs i, i + hd/2) in registers and
// stores the head row into the backbone's cache slot.
#include "fill.cuh"
#include "tc.cuh"

namespace tee {

namespace {

using bf16 = __nv_bfloat16;

constexpr int DKB = 64;            // K per block: one int4 group, one 128-byte swizzle row of bf16
constexpr int RING = 8;            // raw-input slots
constexpr int AHEAD = RING - 2;    // blocks in flight ahead of the one being consumed
constexpr int THREADS_D = 256;
constexpr int MAX_ITEMS = 128;     // MMA M
constexpr uint32_t A_SLOT = MAX_ITEMS * DKB * 2;   // 16 KB

struct DecodeArgs {
    int n_max;
    const int32_t* n_dev;
    int d, kvw, hd, half, group, n_kv;
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
    uint32_t slot_bytes, codes_off, sz_off, g_off;   // layout of one ring slot
};

struct DecodeLayer {
    const uint8_t* wk;
    const uint8_t* wv;
    const __half* k_scale;
    const __half* k_zero;
    const __half* v_scale;
    const __half* v_zero;
    const bf16* gamma;
    int cache_layer;
};

constexpr int MAX_DECODE_LAYERS = 64;
struct DecodeLayers {
    DecodeLayer l[MAX_DECODE_LAYERS];
};

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(tc::smem_u32(dst)), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ float nibble_f32(uint32_t q) {
    // exact small integer as fp32: (2^23 + q) - 2^23
    return __uint_as_float(0x4B000000u | q) - 8388608.0f;
}

__global__ void __launch_bounds__(THREADS_D, 1)
fill_decode_kernel(DecodeArgs a, const __grid_constant__ DecodeLayers layers, void* ws) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int N = a.hd;                                   // columns of this CTA (one head)
    uint8_t* ring = smem;                                 // RING slots of a.slot_bytes
    uint8_t* wb[2] = {smem + RING * a.slot_bytes, smem + RING * a.slot_bytes + N * 128};
    // Small arrays after the operands, widest first so that each stays aligned.
    uint64_t* done = reinterpret_cast<uint64_t*>(wb[1] + N * 128);       // [RING]
    int64_t* s_off = reinterpret_cast<int64_t*>(done + RING);            // [MAX_ITEMS] cache offset or -1
    int* s_row = reinterpret_cast<int*>(s_off + MAX_ITEMS);              // [MAX_ITEMS] source row or -1
    int* s_pos = s_row + MAX_ITEMS;                                      // [MAX_ITEMS]
    float* s_ss = reinterpret_cast<float*>(s_pos + MAX_ITEMS);           // [MAX_ITEMS]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s_ss + MAX_ITEMS);
    int* s_flags = reinterpret_cast<int*>(tmem_slot + 1);                // [0] abort
    volatile int* abort = s_flags;

    const int head2 = blockIdx.x, li = blockIdx.y;
    const DecodeLayer& L = layers.l[li];
    const bool is_k = head2 < a.n_kv;
    const int head = is_k ? head2 : head2 - a.n_kv;
    const int col0 = head * a.hd;
    const uint8_t* codes = is_k ? L.wk : L.wv;
    const __half* scale = is_k ? L.k_scale : L.v_scale;
    const __half* zero = is_k ? L.k_zero : L.v_zero;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = min(item_count(a.n_max, a.n_dev), MAX_ITEMS);
    const uint32_t tmem_cols = N <= 64 ? 64 : 128;
    const int nkb = a.d / DKB;

    if (threadIdx.x == 0) {
        for (int s = 0; s < RING; ++s) tc::mbar_init(&done[s], 1);
        s_flags[0] = 0;
        tc::fence_barrier_init();
    }
    // Per-item metadata: source row, cache offset (validated once per item).
    for (int i = threadIdx.x; i < MAX_ITEMS; i += THREADS_D) {
        int r = -1, p = 0;
        int64_t off = -1;
        if (i < n) {
            r = a.rows ? a.rows[i] : i;
            if (r < 0 || r >= a.h_rows) {
                if (head2 == 0 && li == 0) record_fault(ws, TEE_DEVERR_ROW, r);
                r = -1;
            } else {
                p = a.pos ? a.pos[r] : a.pos0 + r;
                const int sq = a.seq ? a.seq[r] : 0;
                if (!pos_ok(p, a.cl.max_pos, a.hdr)) {
                    if (head2 == 0 && li == 0) record_fault(ws, TEE_DEVERR_POS, p);
                } else if (sq < 0 || sq >= a.cl.n_seq) {
                    if (head2 == 0 && li == 0) record_fault(ws, TEE_DEVERR_SEQ, sq);
                } else {
                    off = L.cache_layer * a.cl.s_layer + sq * a.cl.s_seq + head * a.cl.s_head +
                          static_cast<int64_t>(p) * a.cl.s_pos;
                }
            }
        }
        s_row[i] = r;
        s_pos[i] = p;
        s_off[i] = off;
    }
    if (warp == 0) tc::tmem_alloc(tmem_slot, tmem_cols);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // Issue the cp.async copies of K block kb into its ring slot.
    auto prefetch = [&](int kb) {
        uint8_t* slot = ring + (kb % RING) * a.slot_bytes;
        // A: the item rows x 8 chunks of 16 bytes, swizzled (chunk j of row r at j ^ (r & 7)).
        // Rows from n to 127 were zeroed once and are never written.
        for (int u = threadIdx.x; u < n * 8; u += THREADS_D) {
            const int r = u >> 3, j = u & 7;
            const int src_row = s_row[r];
            const bf16* src = a.h + static_cast<int64_t>(src_row < 0 ? 0 : src_row) * a.ld_h + kb * DKB + j * 8;
            cp_async16(slot + r * 128 + ((j ^ (r & 7)) << 4), src, src_row >= 0);
        }
        // int4 codes: 32 packed rows x N bytes.
        const int cchunks = N / 16;
        for (int u = threadIdx.x; u < 32 * cchunks; u += THREADS_D) {
            const int r = u / cchunks, j = u % cchunks;
            cp_async16(slot + a.codes_off + r * N + j * 16,
                       codes + static_cast<int64_t>(kb * 32 + r) * a.kvw + col0 + j * 16, true);
        }
        // scale and zero of this group (N fp16 each), g_j for these 64 k.
        const int schunks = N * 2 / 16;
        const int64_t gi = static_cast<int64_t>(kb * DKB / a.group) * a.kvw + col0;
        for (int u = threadIdx.x; u < 2 * schunks + 8; u += THREADS_D) {
            if (u < schunks)
                cp_async16(slot + a.sz_off + u * 16, scale + gi + u * 8, true);
            else if (u < 2 * schunks)
                cp_async16(slot + a.sz_off + N * 2 + (u - schunks) * 16, zero + gi + (u - schunks) * 8, true);
            else
                cp_async16(slot + a.g_off + (u - 2 * schunks) * 16, L.gamma + kb * DKB + (u - 2 * schunks) * 8, true);
        }
    };

    // Zero the A rows past the items in every ring slot (the MMA always reads 128 rows).
    for (int u = threadIdx.x; u < RING * (MAX_ITEMS - n) * 8; u += THREADS_D) {
        const int slot = u / ((MAX_ITEMS - n) * 8), rem = u % ((MAX_ITEMS - n) * 8);
        *reinterpret_cast<uint4*>(ring + slot * a.slot_bytes + (n + (rem >> 3)) * 128 + ((rem & 7) << 4)) =
            make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    for (int kb = 0; kb < AHEAD; ++kb) {
        if (kb < nkb) prefetch(kb);
        cp_async_commit();
    }
    float ss = 0.f;                       // partial sum(h^2): item row threadIdx.x >> 1, chunks of one half
    const uint32_t idesc = tc::idesc_bf16(MAX_ITEMS, N);
    bool ok = true;
    for (int kb = 0; kb < nkb; ++kb) {
        // Refill the slot of block kb-2 with block kb+AHEAD once the MMA of kb-2 is done.
        bool w = true;
        if (kb >= 2) w = tc::mbar_wait(&done[(kb - 2) % RING], ((kb - 2) / RING) & 1, abort, ws, 21);
        if (w && kb + AHEAD < nkb) prefetch(kb + AHEAD);
        cp_async_commit();
        cp_async_wait<AHEAD>();           // block kb has landed (this thread's copies)
        if (!__syncthreads_and(w)) {      // ... and everyone else's; leave together on a timeout
            ok = false;
            break;
        }
        const uint8_t* slot = ring + (kb % RING) * a.slot_bytes;
        {
            // Dequantise N columns x 64 k into the B operand: unit = 4 columns x 8 k, all warps.
            const int units = N / 4 * 8;
            for (int u = threadIdx.x; u < units; u += THREADS_D) {
                const int cg = (u >> 5) * 4 + (u & 3);     // column group (4 columns)
                const int kc = (u & 31) >> 2;              // 8 k values
                uint32_t w4[4];
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    w4[r] = *reinterpret_cast<const uint32_t*>(slot + a.codes_off + (4 * kc + r) * N + 4 * cg);
                const uint2 s4 = *reinterpret_cast<const uint2*>(slot + a.sz_off + cg * 8);
                const uint2 z4 = *reinterpret_cast<const uint2*>(slot + a.sz_off + N * 2 + cg * 8);
                const uint4 g8 = *reinterpret_cast<const uint4*>(slot + a.g_off + kc * 16);
                float sc[4], zs[4], g[8];
                unpack_f16x2(s4.x, sc[0], sc[1]);
                unpack_f16x2(s4.y, sc[2], sc[3]);
                unpack_f16x2(z4.x, zs[0], zs[1]);
                unpack_f16x2(z4.y, zs[2], zs[3]);
                unpack_bf16x2(g8.x, g[0], g[1]);
                unpack_bf16x2(g8.y, g[2], g[3]);
                unpack_bf16x2(g8.z, g[4], g[5]);
                unpack_bf16x2(g8.w, g[6], g[7]);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float szj = zs[j] * sc[j];
                    uint32_t packed[4];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const uint32_t byte = (w4[r] >> (8 * j)) & 0xFFu;
                        // (q - z) * s * g  as  (q * s - z * s) * g
                        const float lo = fmaf(nibble_f32(byte & 0xFu), sc[j], -szj) * g[2 * r];
                        const float hi = fmaf(nibble_f32(byte >> 4), sc[j], -szj) * g[2 * r + 1];
                        packed[r] = pack_bf16x2(lo, hi);
                    }
                    const int c = 4 * cg + j;
                    *reinterpret_cast<uint4*>(wb[kb & 1] + c * 128 + ((kc ^ (c & 7)) << 4)) =
                        make_uint4(packed[0], packed[1], packed[2], packed[3]);
                }
            }
            // sum(h^2): two threads per item row, four 16-byte chunks each.
            const int r = threadIdx.x >> 1;
            if (r < n) {
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int j = (threadIdx.x & 1) * 4 + jj;
                    const uint4 v = *reinterpret_cast<const uint4*>(slot + r * 128 + (j << 4));
                    float x[8];
                    unpack_bf16x2(v.x, x[0], x[1]);
                    unpack_bf16x2(v.y, x[2], x[3]);
                    unpack_bf16x2(v.z, x[4], x[5]);
                    unpack_bf16x2(v.w, x[6], x[7]);
#pragma unroll
                    for (int q = 0; q < 8; ++q) ss = fmaf(x[q], x[q], ss);
                }
            }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        if (threadIdx.x == 0) {
            tc::tc_fence_after();
            const uint64_t ad = tc::smem_desc_sw128(tc::smem_u32(slot));
            const uint64_t bd = tc::smem_desc_sw128(tc::smem_u32(wb[kb & 1]));
#pragma unroll
            for (int kk = 0; kk < DKB / 16; ++kk) tc::umma_bf16(tmem, ad + 2 * kk, bd + 2 * kk, idesc, kb | kk);
            tc::umma_commit(&done[kb % RING]);
        }
    }
    cp_async_wait<0>();
    ss += __shfl_xor_sync(0xFFFFFFFFu, ss, 1);
    if ((threadIdx.x & 1) == 0 && (threadIdx.x >> 1) < MAX_ITEMS) s_ss[threadIdx.x >> 1] = ss;
    if (ok && nkb > 0) ok = tc::mbar_wait(&done[(nkb - 1) % RING], ((nkb - 1) / RING) & 1, abort, ws, 22);
    ok = __syncthreads_and(ok);
    tc::tc_fence_after();

    // Epilogue: warps 0-3, thread = item row = TMEM lane, one whole head in its columns.
    if (warp < 4 && ok) {
        const int i = warp * 32 + lane;
        const bool valid = i < n && s_off[i] >= 0;
        const float rs = valid ? 1.0f / sqrtf(s_ss[i] * a.inv_d + a.eps) : 0.f;
        const uint32_t tb = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        bf16* dst = (is_k ? a.kc : a.vc) + (valid ? s_off[i] : 0);
        const float2* cs = a.rope + static_cast<int64_t>(valid ? s_pos[i] : 0) * a.half;
        for (int c = 0; c < a.half; c += 32) {
            float lo[32], hi[32];
            tc::tmem_ld32(tb + c, lo);
            tc::tmem_ld32(tb + a.half + c, hi);
            if (!valid) continue;
            if (is_k) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float2 e = cs[c + j];
                    const float x1 = lo[j] * rs, x2 = hi[j] * rs;
                    lo[j] = x1 * e.x - x2 * e.y;
                    hi[j] = x2 * e.x + x1 * e.y;
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    lo[j] *= rs;
                    hi[j] *= rs;
                }
            }
            uint4* o = reinterpret_cast<uint4*>(dst + c);
            uint4* o2 = reinterpret_cast<uint4*>(dst + a.half + c);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                o[q] = make_uint4(pack_bf16x2(lo[8 * q], lo[8 * q + 1]), pack_bf16x2(lo[8 * q + 2], lo[8 * q + 3]),
                                  pack_bf16x2(lo[8 * q + 4], lo[8 * q + 5]), pack_bf16x2(lo[8 * q + 6], lo[8 * q + 7]));
                o2[q] = make_uint4(pack_bf16x2(hi[8 * q], hi[8 * q + 1]), pack_bf16x2(hi[8 * q + 2], hi[8 * q + 3]),
                                   pack_bf16x2(hi[8 * q + 4], hi[8 * q + 5]), pack_bf16x2(hi[8 * q + 6], hi[8 * q + 7]));
            }
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, tmem_cols);
}

bool decode_eligible(const FillCall& fc) {
    const tee_fill_desc& D = *fc.desc;
    if (D.dtype != TEE_BF16 || D.wfmt != TEE_W_INT4 || D.group != DKB) return false;
    if (fc.n_max > MAX_ITEMS || fc.n_layers > MAX_DECODE_LAYERS) return false;
    if (D.d % DKB || (D.head_dim != 64 && D.head_dim != 128)) return false;
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
    // 16-byte copies of codes rows (kvw bytes apart) and of fp16 scale rows (2*kvw bytes apart)
    const int kvw = D.n_kv_heads * D.head_dim;
    return kvw % 16 == 0;
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
    a.group = D.group;
    a.n_kv = D.n_kv_heads;
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
    // ring slot: A operand (1024-aligned) | codes 32 x N | scale N, zero N (fp16) | g 64 (bf16)
    a.codes_off = A_SLOT;
    a.sz_off = a.codes_off + 32 * a.hd;
    a.g_off = a.sz_off + 4 * a.hd;
    a.slot_bytes = static_cast<uint32_t>(round_up(a.g_off + DKB * 2, 1024));
    DecodeLayers ls{};
    for (int l = 0; l < fc.n_layers; ++l) {
        const tee_fill_layer& L = fc.layers[l];
        ls.l[l] = DecodeLayer{static_cast<const uint8_t*>(L.wk), static_cast<const uint8_t*>(L.wv),
                              static_cast<const __half*>(L.k_scale), static_cast<const __half*>(L.k_zero),
                              static_cast<const __half*>(L.v_scale), static_cast<const __half*>(L.v_zero),
                              static_cast<const bf16*>(L.gamma), L.cache_layer};
    }
    // alignment slack | ring | two B buffers | small arrays (see the kernel's layout)
    const size_t small = RING * 8 + MAX_ITEMS * (8 + 4 + 4 + 4) + 4 + 4 * 4;
    const size_t smem = 1024 + RING * size_t(a.slot_bytes) + 2 * size_t(a.hd) * 128 + round_up(small, 16);
    tee_status st = cuda_status(
        cudaFuncSetAttribute(fill_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)));
    if (st != TEE_OK) return st;
    dim3 grid(2 * D.n_kv_heads, fc.n_layers);
    fill_decode_kernel<<<grid, THREADS_D, smem, fc.stream>>>(a, ls, fc.ws);
    return launch_status();
}

}  // namespace tee
