// The front of a decode step in one launch: River-LLM's cosine gate (background
// "state transition similarity"; method step 3), TIDE's batch compaction and
// exit scatter (core module 4), for batches of up to 128 tokens.
//
// One cluster of C <= 8 CTAs of W = ceil(n / 8) warps (W <= 16), a warp per
// token, so that even a small batch spreads over eight SMs. Each warp
// streams its token's rows of h_prev and h_cur (16-byte loads, eight chunks of
// each row per lane in flight; the h_cur chunks stay in registers), reduces
// <a,b>, |a|^2, |b|^2 in fp32 and forms the score. Each CTA publishes, in its
// shared memory, the minimum score of its tokens and how many of them exit on
// their own; after one cluster barrier every CTA reads the C pairs through
// distributed shared memory: the batch minimum gives the all-tokens flag (the
// batch rule's mask), the counts give each CTA's offset in the stable split.
// Every warp then writes its token's mask, list entry and position, and stores
// its h_cur row from registers: to its slot of `out` if it exits (the scatter),
// to its place in h_cont if it continues (the gather). A second cluster
// barrier keeps every CTA's shared memory alive until all reads are done.
// The results equal tee_exit_gate followed by tee_exit_compact_scatter.
#include <type_traits>

#include "common.cuh"

namespace tee {

namespace {

constexpr int FW = 16;                 // warps (tokens) per CTA at most
constexpr int F_THREADS = FW * 32;
constexpr int F_MAX_CTAS = 8;          // portable cluster size
constexpr int F_MAX_TOKENS = FW * F_MAX_CTAS;
constexpr int F_KEEP = 8;              // 16-byte chunks of a row per lane kept in registers

struct FrontArgs {
    int n, d, rule;
    float thr;
    const void* h_cur;
    int64_t ld_cur;
    const void* h_prev;
    int64_t ld_prev;
    const int32_t* pos_in;
    float* score;
    uint8_t* mask;
    int32_t* flag;
    int32_t* cont_rows;
    int32_t* exit_rows;
    int32_t* cont_pos;
    int32_t* exit_pos;
    void* h_cont;
    int64_t ld_cont;
    void* out;
    int64_t ld_out;
    int64_t n_out;
    int32_t* counts;
    void* ws;
};

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
// 32-bit word at shared-memory address `saddr` of cluster CTA `cta`.
__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t saddr, uint32_t cta) {
    uint32_t remote, v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(saddr), "r"(cta));
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(remote) : "memory");
    return v;
}
__device__ __forceinline__ uint4 ld_row16(const void* p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
template <typename T>
__device__ __forceinline__ void cos_acc16(uint4 a, uint4 b, float& dot, float& na, float& nb) {
    const uint32_t ua[4] = {a.x, a.y, a.z, a.w}, ub[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        if constexpr (sizeof(T) == 4) {
            const float x = __uint_as_float(ua[q]), y = __uint_as_float(ub[q]);
            dot = fmaf(x, y, dot);
            na = fmaf(x, x, na);
            nb = fmaf(y, y, nb);
        } else {
            float x0, x1, y0, y1;
            if constexpr (std::is_same<T, __half>::value) {
                unpack_f16x2(ua[q], x0, x1);
                unpack_f16x2(ub[q], y0, y1);
            } else {
                unpack_bf16x2(ua[q], x0, x1);
                unpack_bf16x2(ub[q], y0, y1);
            }
            dot = fmaf(x0, y0, dot);
            dot = fmaf(x1, y1, dot);
            na = fmaf(x0, x0, na);
            na = fmaf(x1, x1, na);
            nb = fmaf(y0, y0, nb);
            nb = fmaf(y1, y1, nb);
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(F_THREADS, 1) front_kernel(const __grid_constant__ FrontArgs a) {
    __shared__ float s_score[FW];
    __shared__ uint32_t s_pub[2];       // this CTA's minimum score (bits) and its tokens exiting on their own
    __shared__ uint32_t s_exit_bits;    // bit w: token of warp w exits on its own
    allow_dependents();
    wait_prior_grid();   // launched as a dependent (a copy kernel before it): every access waits for it
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t cta = cluster_rank();
    const int n_ctas = static_cast<int>(gridDim.x);   // the grid is one cluster
    const int fw = static_cast<int>(blockDim.x) >> 5;   // tokens per CTA
    const int t = static_cast<int>(cta) * fw + warp;
    const bool live = t < a.n;
    constexpr int V = 16 / sizeof(T);
    const int nch = a.d / V;
    const T* hc = static_cast<const T*>(a.h_cur) + static_cast<int64_t>(live ? t : 0) * a.ld_cur;
    const T* hp = static_cast<const T*>(a.h_prev) + static_cast<int64_t>(live ? t : 0) * a.ld_prev;
    const int p = (live && a.pos_in) ? a.pos_in[t] : t;   // the token's slot, fetched early

    // ---- score: the first 32 * F_KEEP chunks of both rows in flight at once,
    // h_cur's kept for the copy; longer rows stream the rest.
    uint4 keep[F_KEEP];
    float dot = 0.f, na = 0.f, nb = 0.f;
    {
        uint4 xa[F_KEEP];
#pragma unroll
        for (int u = 0; u < F_KEEP; ++u) {
            const int c = lane + 32 * u;
            const bool in = live && c < nch;
            xa[u] = in ? ld_row16(hp + c * V) : make_uint4(0u, 0u, 0u, 0u);
            keep[u] = in ? ld_row16(hc + c * V) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < F_KEEP; ++u) cos_acc16<T>(xa[u], keep[u], dot, na, nb);
    }
    if (live)
        for (int c0 = 32 * F_KEEP + lane; c0 < nch; c0 += 32 * F_KEEP) {
            uint4 ya[F_KEEP], yb[F_KEEP];
#pragma unroll
            for (int u = 0; u < F_KEEP; ++u) {
                const int c = c0 + 32 * u;
                ya[u] = c < nch ? ld_row16(hp + c * V) : make_uint4(0u, 0u, 0u, 0u);
                yb[u] = c < nch ? ld_row16(hc + c * V) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < F_KEEP; ++u) cos_acc16<T>(ya[u], yb[u], dot, na, nb);
        }
    dot = warp_sum(dot);
    na = warp_sum(na);
    nb = warp_sum(nb);
    const float den = sqrtf(na) * sqrtf(nb);
    const float s = den > 0.f ? dot / den : 0.f;
    if (lane == 0) {
        s_score[warp] = s;
        if (live) a.score[t] = s;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float m = INFINITY;
        uint32_t bits = 0;
        for (int w = 0; w < fw; ++w) {
            if (static_cast<int>(cta) * fw + w >= a.n) break;
            const float sw = s_score[w];
            m = fminf(m, sw == sw ? sw : -INFINITY);   // a NaN score never lets the batch exit
            if (exits(sw, a.thr)) bits |= 1u << w;
        }
        s_pub[0] = __float_as_uint(m);
        s_pub[1] = static_cast<uint32_t>(__popc(bits));
        s_exit_bits = bits;
    }
    cluster_arrive_release();   // publish s_pub to the cluster
    cluster_wait();

    // ---- the batch: minimum score and the exits of the CTAs before this one
    float gmin = INFINITY;
    int before = 0, total = 0;
    const uint32_t pub = static_cast<uint32_t>(__cvta_generic_to_shared(s_pub));
    for (int c = 0; c < n_ctas; ++c) {
        const float mc = __uint_as_float(ld_cluster_u32(pub, static_cast<uint32_t>(c)));
        const int kc = static_cast<int>(ld_cluster_u32(pub + 4, static_cast<uint32_t>(c)));
        gmin = fminf(gmin, mc);
        total += kc;
        if (c < static_cast<int>(cta)) before += kc;
    }
    cluster_arrive_release();   // done with the other CTAs' shared memory (they wait before leaving);
                                // release: those loads are complete before the arrival counts
    const bool all_exit = a.n > 0 && gmin > a.thr;
    uint32_t bits = s_exit_bits;
    if (a.rule == TEE_RULE_BATCH_ALL) {
        const int live_here = min(max(a.n - static_cast<int>(cta) * fw, 0), fw);
        bits = all_exit ? (1u << live_here) - 1u : 0u;   // live_here <= 16
        before = all_exit ? min(static_cast<int>(cta) * fw, a.n) : 0;
        total = all_exit ? a.n : 0;
    }
    const bool ex = live && ((bits >> warp) & 1u);
    const int e_idx = before + __popc(bits & ((1u << warp) - 1u));   // exiting tokens before t
    const int c_idx = t - e_idx;                                    // continuing tokens before t
    if (lane == 0 && live) {
        a.mask[t] = ex ? 1 : 0;
        if (ex) {
            a.exit_rows[e_idx] = t;
            if (a.exit_pos) a.exit_pos[e_idx] = p;
        } else {
            a.cont_rows[c_idx] = t;
            if (a.cont_pos) a.cont_pos[c_idx] = p;
        }
    }
    if (cta == 0 && threadIdx.x == 0) {
        a.counts[0] = a.n - total;
        a.counts[1] = total;
        if (a.flag) *a.flag = all_exit ? 1 : 0;
    }

    // ---- the token's row: scattered to its slot if it exits, gathered if it continues
    if (live) {
        T* dst = nullptr;
        if (ex) {
            if (a.out) {
                if (p < 0 || p >= a.n_out) {
                    if (lane == 0) record_fault(a.ws, TEE_DEVERR_DEST, p);
                } else {
                    dst = static_cast<T*>(a.out) + static_cast<int64_t>(p) * a.ld_out;
                }
            }
        } else if (a.h_cont) {
            dst = static_cast<T*>(a.h_cont) + static_cast<int64_t>(c_idx) * a.ld_cont;
        }
        if (dst) {
#pragma unroll
            for (int u = 0; u < F_KEEP; ++u) {
                const int c = lane + 32 * u;
                if (c < nch) *reinterpret_cast<uint4*>(dst + c * V) = keep[u];
            }
            for (int c = 32 * F_KEEP + lane; c < nch; c += 32)
                *reinterpret_cast<uint4*>(dst + c * V) = ld_row16(hc + c * V);
        }
    }
    cluster_wait();   // no CTA leaves while another may still read its s_pub
}

template <typename T>
tee_status launch_front(const FrontArgs& a, cudaStream_t stream) {
    const int fw = (a.n + F_MAX_CTAS - 1) / F_MAX_CTAS;   // 1..16 tokens per CTA
    const int ctas = (a.n + fw - 1) / fw;                 // <= 8
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(fw * 32);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ctas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // it may start launching while the kernel before it runs (it waits for that
    // kernel before any memory access)
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    const tee_status st = cuda_status(cudaLaunchKernelEx(&cfg, front_kernel<T>, a));
    return st != TEE_OK ? st : launch_status();
}

}  // namespace

}  // namespace tee

using namespace tee;

extern "C" size_t tee_exit_gate_compact_scatter_workspace_size(const tee_gate_desc* g, int32_t n) {
    if (!g || n < 0) return 0;
    const size_t a = tee_exit_gate_workspace_size(g, n), b = tee_exit_compact_workspace_size(n);
    return a > b ? a : b;
}

extern "C" tee_status tee_exit_gate_compact_scatter(const tee_gate_desc* g, int32_t n, const void* h_cur,
                                                    int64_t ld_cur, const void* h_prev, int64_t ld_prev,
                                                    const void* gamma, const void* w_down, const float* b_down,
                                                    const void* w_up, const float* b_up, const int32_t* pos_in,
                                                    float* score, uint8_t* mask, int32_t* batch_flag,
                                                    int32_t* cont_rows, int32_t* exit_rows, int32_t* cont_pos,
                                                    int32_t* exit_pos, void* h_cont, int64_t ld_cont, void* out,
                                                    int64_t ld_out, int64_t n_out, int32_t* counts, void* ws,
                                                    size_t ws_bytes, void* stream) {
    if (!g || n < 0 || !counts) return TEE_ERR_INVALID_ARG;
    if (!ws || ws_bytes < tee_exit_gate_compact_scatter_workspace_size(g, n)) return TEE_ERR_WORKSPACE;
    const size_t es = dtype_bytes(g->dtype);
    if (es == 0) return TEE_ERR_UNSUPPORTED;
    if (n > 0 && (!h_cur || !out || !cont_rows || !exit_rows || !score || !mask)) return TEE_ERR_INVALID_ARG;
    if (n > 0 && (n_out < 0 || ld_out < g->d || (ld_out * es) % 16 || !aligned16(out))) return TEE_ERR_INVALID_ARG;
    if (n > 0 && h_cont && (ld_cont < g->d || (ld_cont * es) % 16 || !aligned16(h_cont))) return TEE_ERR_INVALID_ARG;
    const bool one_launch = g->mode == TEE_GATE_COSINE && n >= 1 && n <= F_MAX_TOKENS;
    if (!one_launch) {   // the two calls it stands for
        tee_status st = tee_exit_gate(g, n, h_cur, ld_cur, h_prev, ld_prev, gamma, w_down, b_down, w_up, b_up,
                                      score, mask, batch_flag, ws, ws_bytes, stream);
        if (st != TEE_OK) return st;
        return tee_exit_compact_scatter(n, mask, pos_in, h_cur, ld_cur, g->d, g->dtype, cont_rows, exit_rows,
                                        cont_pos, exit_pos, h_cont, ld_cont, out, ld_out, n_out, counts, ws,
                                        ws_bytes, stream);
    }
    // the same checks as the gate's cosine path
    if (g->d <= 0 || g->d % 8 != 0 || !(g->threshold == g->threshold)) return TEE_ERR_INVALID_ARG;
    if (g->rule != TEE_RULE_PER_TOKEN && g->rule != TEE_RULE_BATCH_ALL) return TEE_ERR_INVALID_ARG;
    if (!h_prev || ld_cur < g->d || ld_prev < g->d || (ld_cur * es) % 16 || (ld_prev * es) % 16 ||
        !aligned16(h_cur) || !aligned16(h_prev))
        return TEE_ERR_INVALID_ARG;
    FrontArgs a{};
    a.n = n;
    a.d = g->d;
    a.rule = g->rule;
    a.thr = g->threshold;
    a.h_cur = h_cur;
    a.ld_cur = ld_cur;
    a.h_prev = h_prev;
    a.ld_prev = ld_prev;
    a.pos_in = pos_in;
    a.score = score;
    a.mask = mask;
    a.flag = batch_flag;
    a.cont_rows = cont_rows;
    a.exit_rows = exit_rows;
    a.cont_pos = cont_pos;
    a.exit_pos = exit_pos;
    a.h_cont = h_cont;
    a.ld_cont = ld_cont;
    a.out = out;
    a.ld_out = ld_out;
    a.n_out = n_out;
    a.counts = counts;
    a.ws = ws;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (g->dtype) {
        case TEE_F32: return launch_front<float>(a, s);
        case TEE_F16: return launch_front<__half>(a, s);
        default: return launch_front<__nv_bfloat16>(a, s);
    }
}
